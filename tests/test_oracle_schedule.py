"""Pins of the oracle's schedule (chunks, Gamma(i), history, slots, Tail_H)
against the facts of the FlashForward pages and hand-worked tables."""
import os

import numpy as np
import pytest

from oracle import ff_oracle as fo

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLD, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_81_latents_make_27_chunks_of_3():
    # onedev.kr/papers/332 "무엇과 다른가": 81 positions -> 27 chunks of 3 latents.
    assert fo.num_chunks(81, 3) == 27
    covered = []
    for i in range(27):
        s, e = fo.chunk_span(i, 3, 81)
        assert e - s + 1 == 3
        covered.extend(range(s, e + 1))
    assert covered == list(range(81))
    with pytest.raises(ValueError):
        fo.chunk_span(27, 3, 81)


def test_gamma_table_81():
    rows = _rows("gamma_81.txt")
    assert len(rows) == 27
    for r in rows:
        i, s, e, left, right = map(int, r)
        assert fo.chunk_span(i, 3, 81) == (s, e)
        assert fo.gamma(i, 3, 10, 81) == [left, right]


def test_anchor_set_and_planner_blocks():
    # Anchors at {0,10,...,80}: 9 of them, produced 3 per planner block.
    used = sorted({a for i in range(27) for a in fo.gamma(i, 3, 10, 81)})
    assert used == list(range(0, 81, 10))
    blocks = [used[j:j + 3] for j in range(0, 9, 3)]
    assert blocks == [[0, 10, 20], [30, 40, 50], [60, 70, 80]]
    # every chunk's anchors lie in at most two consecutive planner blocks
    for i in range(27):
        g = fo.gamma(i, 3, 10, 81)
        assert max(g) // 30 - min(g) // 30 <= 1


def test_context_budget_w_ctx():
    # W_ctx = 21 latent frames; context = anchors + H chunks of history + own chunk.
    H, BR = 5, 3
    key_frames = []
    for i in range(27):
        n = len(fo.gamma(i, BR, 10, 81)) + BR * len(fo.history_chunks(i, H)) + BR
        key_frames.append(n)
        assert n <= 21
    assert key_frames[:6] == [5, 8, 11, 14, 17, 20]
    assert max(key_frames) == 20
    assert sum(key_frames) == 495


def test_tiny_table():
    rows = _rows("tiny_schedule.txt")
    assert fo.num_chunks(13, 3) == len(rows) == 5
    for r in rows:
        i, s, e = int(r[0]), int(r[1]), int(r[2])
        anchors = [int(x) for x in r[3].split(",")]
        hist_f, own_f, key_f, slot = map(int, r[4:])
        assert fo.chunk_span(i, 3, 13) == (s, e)
        assert fo.gamma(i, 3, 4, 13) == anchors
        hist = fo.history_chunks(i, 2)
        hf = sum(fo.chunk_span(j, 3, 13)[1] - fo.chunk_span(j, 3, 13)[0] + 1 for j in hist)
        assert hf == hist_f
        assert e - s + 1 == own_f
        assert len(anchors) + hist_f + own_f == key_f
        assert fo.bank_slot(i, 2) == slot


def test_gamma_edge_rules():
    # right anchor past the last latent is dropped (stride 10, 75 latents: chunk 24 = [72,74] -> right 80 > 74)
    assert fo.gamma(24, 3, 10, 75) == [70]
    # coincident anchors used once
    assert fo.gamma(4, 3, 4, 13) == [12]
    # chunk ending exactly on an anchor
    assert fo.gamma(6, 3, 10, 81) == [10, 20]
    # 261 latents: every right anchor exists
    for i in range(87):
        assert len(fo.gamma(i, 3, 10, 261)) == 2


def _tiny_cfg(**kw):
    base = dict(n_layers=1, total_frames=13, heads=1, head_dim=8, frame_h=1, frame_w=2,
                n_stages=1, history=2, chunk_frames=3, anchor_stride=4, anchor_capacity=4)
    base.update(kw)
    return fo.BankConfig(**base)


def _zeros(cfg, frames):
    return np.zeros((frames * cfg.tokens_per_frame, cfg.heads, cfg.head_dim), np.uint16)


def test_tail_h_tags_over_rollout():
    # Eq. (2): after chunk i the stage bank holds exactly chunks max(0, i-H+1) .. i.
    for H in (1, 2, 5):
        cfg = _tiny_cfg(total_frames=81, history=H, anchor_stride=10, anchor_capacity=9)
        bank = fo.OracleBank(cfg)
        for a0 in (0, 30, 60):
            bank.anchor_publish(0, a0, 3, _zeros(cfg, 3), _zeros(cfg, 3))
        for i in range(27):
            s, e = fo.chunk_span(i, 3, 81)
            res = bank.render(0, 0, i, _zeros(cfg, e - s + 1), _zeros(cfg, e - s + 1), _zeros(cfg, e - s + 1))
            tags = sorted(t for t in bank.stage_tags(0, 0) if t >= 0)
            assert tags == list(range(max(0, i - H + 1), i + 1))
            assert res.history == list(range(max(0, i - H), i))


def test_context_reads_slot_before_overwrite():
    # With H = 2, chunk 2 publishes into the slot that holds chunk 0, which chunk 2 still attends to.
    cfg = _tiny_cfg()
    bank = fo.OracleBank(cfg)
    bank.anchor_publish(0, 0, 4, _zeros(cfg, 4), _zeros(cfg, 4))
    for i in range(5):
        s, e = fo.chunk_span(i, 3, 13)
        res = bank.render(0, 0, i, _zeros(cfg, e - s + 1), _zeros(cfg, e - s + 1), _zeros(cfg, e - s + 1))
        if i == 2:
            assert res.context_frames == [4, 8, 0, 1, 2, 3, 4, 5, 6, 7, 8]
        if i == 4:
            assert res.context_frames == [12, 6, 7, 8, 9, 10, 11, 12]


def test_order_and_anchor_errors():
    cfg = _tiny_cfg()
    bank = fo.OracleBank(cfg)
    z3 = _zeros(cfg, 3)
    with pytest.raises(fo.OracleError) as ei:
        bank.render(0, 0, 0, z3, z3, z3)
    assert ei.value.code == "FF_ERR_ANCHOR_MISSING"
    bank.anchor_publish(0, 0, 2, _zeros(cfg, 2), _zeros(cfg, 2))
    with pytest.raises(fo.OracleError) as ei:
        bank.render(0, 0, 1, z3, z3, z3)
    assert ei.value.code == "FF_ERR_ORDER"
    bank.render(0, 0, 0, z3, z3, z3)
    with pytest.raises(fo.OracleError) as ei:
        bank.render(0, 0, 1, z3, z3, z3)   # needs anchor 8, not yet published
    assert ei.value.code == "FF_ERR_ANCHOR_MISSING"
    with pytest.raises(fo.OracleError):
        bank.anchor_publish(0, 2, 1, _zeros(cfg, 1), _zeros(cfg, 1))  # not on the stride


def test_anchor_ring_capacity_6_covers_261_latent_rollout():
    # Reading for long rollouts: publish planner block j (anchors 30j, 30j+10, 30j+20) just
    # before the first chunk that needs one of them; a 6-slot anchor ring then never evicts
    # an anchor that a later chunk still needs.
    cfg = _tiny_cfg(total_frames=261, history=5, anchor_stride=10, anchor_capacity=6)
    bank = fo.OracleBank(cfg)
    published = set()
    for i in range(87):
        for a in fo.gamma(i, 3, 10, 261):
            blk = a // 30
            if blk not in published:
                n = min(3, (260 - 30 * blk) // 10 + 1)
                bank.anchor_publish(0, 30 * blk, n, _zeros(cfg, n), _zeros(cfg, n))
                published.add(blk)
        bank.render(0, 0, i, _zeros(cfg, 3), _zeros(cfg, 3), _zeros(cfg, 3))
    assert len(published) == 9


def test_tiny_bank_render_equals_bruteforce_over_named_frames():
    # The bank's context must be exactly: Gamma(i) anchors (rotated at their own frame),
    # the last H same-stage chunks (rotated at their frames) and the chunk itself.
    cfg = _tiny_cfg(heads=2, head_dim=12, frame_h=1, frame_w=2, n_stages=2)
    T = cfg.tokens_per_frame
    rng = np.random.default_rng(21)
    bits = lambda n: fo.f64_to_bf16_bits(rng.standard_normal((n * T, cfg.heads, cfg.head_dim)))
    bank = fo.OracleBank(cfg)
    anchor_k, anchor_v = bits(4), bits(4)
    bank.anchor_publish(0, 0, 4, anchor_k, anchor_v)
    seen = {0: {}, 1: {}}   # stage -> frame -> (k_bits, v_bits)
    for i in range(5):
        for st in range(2):
            s, e = fo.chunk_span(i, 3, 13)
            nf = e - s + 1
            q, k, v = bits(nf), bits(nf), bits(nf)
            res = bank.render(0, st, i, q, k, v)
            for r, f in enumerate(range(s, e + 1)):
                seen[st][f] = (k[r * T:(r + 1) * T], v[r * T:(r + 1) * T])
            frames_k, frames_v = [], []
            for a in fo.gamma(i, 3, 4, 13):
                j = a // 4
                pos = fo.token_positions([a], 1, 2)
                frames_k.append(fo.rope_k_bits(anchor_k[j * T:(j + 1) * T], pos, 12, 1e4))
                frames_v.append(anchor_v[j * T:(j + 1) * T])
            for f in range(3 * max(0, i - 2), e + 1):
                pos = fo.token_positions([f], 1, 2)
                frames_k.append(fo.rope_k_bits(seen[st][f][0], pos, 12, 1e4))
                frames_v.append(seen[st][f][1])
            K = fo.bf16_bits_to_f64(np.concatenate(frames_k))
            V = fo.bf16_bits_to_f64(np.concatenate(frames_v))
            Q = fo.rope_q_f64(q, fo.token_positions(list(range(s, e + 1)), 1, 2), 12, 1e4)
            bf = np.array(fo.attention_bruteforce(Q.tolist(), K.tolist(), V.tolist()))
            assert np.allclose(res.out, bf, atol=1e-12, rtol=0)
            assert res.key_frames == len(frames_k)


def test_planner_blocks_and_w_ctx():
    # onedev.kr/papers/332 "무엇과 다른가": 9 anchors produced 3 at a time; planner history
    # H_P = 6 and context budget W_ctx = 21 = 6 * 3 + 3.
    assert fo.num_planner_blocks(81, 10, 3) == 3
    assert [fo.planner_block_anchors(b, 3, 10, 81) for b in range(3)] == [[0, 10, 20], [30, 40, 50], [60, 70, 80]]
    assert fo.num_planner_blocks(261, 10, 3) == 9
    widths = []
    for b in range(9):
        hist = fo.planner_history_blocks(b, 6)
        frames = [a for hb in hist for a in fo.planner_block_anchors(hb, 3, 10, 261)]
        frames += fo.planner_block_anchors(b, 3, 10, 261)
        widths.append(len(frames))
        if b == 8:
            assert frames == list(range(60, 261, 10))
    assert max(widths) == 21 and widths == [3, 6, 9, 12, 15, 18, 21, 21, 21]
    # 13 latents at stride 4: anchors {0,4,8,12}, blocks {0,4,8} and {12}
    assert [fo.planner_block_anchors(b, 3, 4, 13) for b in range(2)] == [[0, 4, 8], [12]]
    with pytest.raises(ValueError):
        fo.planner_block_anchors(2, 3, 4, 13)


def test_planner_attention_equals_bruteforce_over_named_frames():
    cfg = _tiny_cfg(heads=2, head_dim=12, frame_h=1, frame_w=2, total_frames=13, anchor_stride=4, anchor_capacity=4)
    T = cfg.tokens_per_frame
    rng = np.random.default_rng(31)
    bits = lambda n: fo.f64_to_bf16_bits(rng.standard_normal((n * T, cfg.heads, cfg.head_dim)))
    bank = fo.OracleBank(cfg)
    ak, av = bits(3), bits(3)
    bank.anchor_publish(0, 0, 3, ak, av)          # clean KV of block 0 = anchors 0, 4, 8
    q, k, v = bits(1), bits(1), bits(1)           # block 1 = anchor 12
    out, frames = bank.planner_attn(0, 1, q, k, v, planner_block=3, planner_history=6)
    assert frames == [0, 4, 8, 12]
    Ks = [fo.rope_k_bits(ak[j * T:(j + 1) * T], fo.token_positions([4 * j], 1, 2), 12, 1e4) for j in range(3)]
    Ks.append(fo.rope_k_bits(k, fo.token_positions([12], 1, 2), 12, 1e4))
    K = fo.bf16_bits_to_f64(np.concatenate(Ks))
    V = fo.bf16_bits_to_f64(np.concatenate([av, v]))
    Q = fo.rope_q_f64(q, fo.token_positions([12], 1, 2), 12, 1e4)
    bf = np.array(fo.attention_bruteforce(Q.tolist(), K.tolist(), V.tolist()))
    assert np.allclose(out, bf, atol=1e-12, rtol=0)
    with pytest.raises(fo.OracleError):
        fo.OracleBank(cfg).planner_attn(0, 1, q, k, v, planner_block=3, planner_history=6)


def test_packed_block_causal_equals_masked_attention_bruteforce():
    # The packed forward is the sequential renderer at one stage; check it against a
    # brute-force attention over all packed tokens with the block mask written out
    # (chunk i sees anchors Gamma(i), chunks i-H..i-1 and itself).
    cfg = _tiny_cfg(heads=1, head_dim=12, frame_h=1, frame_w=2, total_frames=13, anchor_stride=4, anchor_capacity=4)
    T, N, H = cfg.tokens_per_frame, 13, cfg.history
    rng = np.random.default_rng(41)
    bits = lambda n: fo.f64_to_bf16_bits(rng.standard_normal((n * T, 1, 12)))
    q, k, v = bits(N), bits(N), bits(N)
    ak, av = bits(4), bits(4)
    got = fo.packed_block_causal(cfg, q, k, v, ak, av)
    # all keys: anchors (rotated at their frames) then frames (rotated at theirs)
    Ka = np.concatenate([fo.rope_k_bits(ak[j * T:(j + 1) * T], fo.token_positions([4 * j], 1, 2), 12, 1e4)
                         for j in range(4)])
    Kf = fo.rope_k_bits(k, fo.token_positions(list(range(N)), 1, 2), 12, 1e4)
    K = fo.bf16_bits_to_f64(np.concatenate([Ka, Kf]))[:, 0]
    V = fo.bf16_bits_to_f64(np.concatenate([av, v]))[:, 0]
    Q = fo.rope_q_f64(q, fo.token_positions(list(range(N)), 1, 2), 12, 1e4)[:, 0]
    key_frame = [4 * j for j in range(4) for _ in range(T)] + [f for f in range(N) for _ in range(T)]
    is_anchor = [True] * (4 * T) + [False] * (N * T)
    for row in range(N * T):
        f = row // T
        i = f // 3
        s, e = fo.chunk_span(i, 3, N)
        g = fo.gamma(i, 3, 4, N)
        lo = 3 * max(0, i - H)
        allowed = [j for j in range(len(key_frame))
                   if (is_anchor[j] and key_frame[j] in g) or (not is_anchor[j] and lo <= key_frame[j] <= e)]
        ref = fo.attention_bruteforce([[Q[row].tolist()]], [[K[j].tolist()] for j in allowed],
                                      [[V[j].tolist()] for j in allowed])
        assert np.allclose(got[row, 0], ref[0][0], atol=1e-12)
