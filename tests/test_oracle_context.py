"""Pins of the oracle's split form of a renderer call: ``render_context`` (the
context assembly without the attention) and ``commit_publish`` (the bank
update alone), and of ``token_positions``.

The large-shape GPU tests evaluate the attention definition on sampled rows of
``render_context``'s output and keep the oracle's bank in step with
``commit_publish``, so both are tied here to ``render``, which is itself pinned
against a brute force over explicitly named frames
(test_oracle_schedule.py).  Source: FlashForward, onedev.kr/papers/332,
section "어떻게 동작하나", Eq. (2): chunk i reads B_k^(i) (anchors of Gamma(i),
the last H same-stage chunks) and then leaves B_k^(i+1) = Tail_H(B_k^(i) U (i, K, V)).
"""
import math

import numpy as np
import pytest

from oracle import ff_oracle as fo


def _cfg(**kw):
    base = dict(n_layers=1, total_frames=13, heads=2, head_dim=12, frame_h=2, frame_w=3,
                n_stages=2, history=2, chunk_frames=3, anchor_stride=4, anchor_capacity=4)
    base.update(kw)
    return fo.BankConfig(**base)


# tiny config of the renderer (13 latents, stride 4, H 2), then small descriptions
# with H = 1, a short final chunk, an anchor ring that wraps (capacity below the
# anchor count, blocks published on demand) and B_R = 1 / 2
CASES = [
    dict(),
    dict(history=1),
    dict(history=3, total_frames=17, chunk_frames=2, anchor_stride=3, anchor_capacity=3),
    dict(history=2, total_frames=31, chunk_frames=3, anchor_stride=5, anchor_capacity=3),
    dict(history=4, total_frames=11, chunk_frames=1, anchor_stride=2, anchor_capacity=6, n_stages=1),
]


def _publish_needed(banks, cfg, i, published, rng_bits):
    """Publish every anchor of Gamma(i) that is not resident, identically into all banks."""
    for a in fo.gamma(i, cfg.chunk_frames, cfg.anchor_stride, cfg.total_frames):
        sl = banks[0].anchor[0][fo.anchor_slot(a, cfg.anchor_stride, cfg.anchor_capacity)]
        if sl.tag == a:
            continue
        kb, vb = rng_bits(1), rng_bits(1)
        for b in banks:
            b.anchor_publish(0, a, 1, kb, vb)
        published.append(a)


def _slot_state(bank, stage):
    return [(sl.tag, sl.frames, None if sl.k is None else sl.k.tobytes(),
             None if sl.v is None else sl.v.tobytes()) for sl in bank.stage[0][stage]]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_render_context_and_commit_publish_equal_render(case):
    cfg = _cfg(**CASES[case])
    T = cfg.tokens_per_frame
    rng = np.random.default_rng(100 + case)
    bits = lambda n: fo.f64_to_bf16_bits(rng.standard_normal((n * T, cfg.heads, cfg.head_dim)))
    whole = fo.OracleBank(cfg)    # advanced by render()
    split = fo.OracleBank(cfg)    # advanced by render_context() + commit_publish()
    published = []
    for i in range(fo.num_chunks(cfg.total_frames, cfg.chunk_frames)):
        _publish_needed([whole, split], cfg, i, published, bits)
        s, e = fo.chunk_span(i, cfg.chunk_frames, cfg.total_frames)
        nf = e - s + 1
        for st in range(cfg.n_stages):
            q, k, v = bits(nf), bits(nf), bits(nf)
            Q, K, V, k_rot = split.render_context(0, st, i, q, k, v)
            # render_context changes no state
            assert split.next_chunk[0][st] == i
            res = whole.render(0, st, i, q, k, v)
            assert K.shape[0] == V.shape[0] == res.key_frames * T
            np.testing.assert_allclose(fo.attention_f64(Q, K, V), res.out, rtol=0, atol=1e-12)
            assert np.array_equal(k_rot, res.k_rot_bits)
            split.commit_publish(0, st, i, k_rot, v)
            assert _slot_state(split, st) == _slot_state(whole, st)
            assert split.next_chunk == whole.next_chunk
    if cfg.anchor_capacity < fo.num_anchors(cfg.total_frames, cfg.anchor_stride):
        assert len(published) > cfg.anchor_capacity  # the anchor ring wrapped


def test_render_context_rejects_a_stale_history_slot():
    # A history slot that does not carry its chunk's tag must not reach the reference.
    cfg = _cfg(n_stages=1)
    T = cfg.tokens_per_frame
    z = lambda n: np.zeros((n * T, cfg.heads, cfg.head_dim), np.uint16)
    bank = fo.OracleBank(cfg)
    bank.anchor_publish(0, 0, 4, z(4), z(4))
    for i in range(2):
        bank.render(0, 0, i, z(3), z(3), z(3))
    bank.stage[0][0][fo.bank_slot(0, cfg.history)].tag = 7   # corrupt chunk 0's slot
    with pytest.raises(AssertionError):
        bank.render_context(0, 0, 2, z(3), z(3), z(3))


def test_render_context_error_codes_match_render():
    cfg = _cfg(n_stages=1)
    T = cfg.tokens_per_frame
    z = lambda n: np.zeros((n * T, cfg.heads, cfg.head_dim), np.uint16)
    bank = fo.OracleBank(cfg)
    with pytest.raises(fo.OracleError) as ei:
        bank.render_context(0, 0, 0, z(3), z(3), z(3))
    assert ei.value.code == "FF_ERR_ANCHOR_MISSING"
    bank.anchor_publish(0, 0, 2, z(2), z(2))
    with pytest.raises(fo.OracleError) as ei:
        bank.render_context(0, 0, 1, z(3), z(3), z(3))
    assert ei.value.code == "FF_ERR_ORDER"


def test_token_positions_hand_values():
    # (t, y, x) of token n of latent frame f: t = f, frames row-major over (y, x).
    p = fo.token_positions([7], 4, 4)
    assert p.shape == (16, 3)
    assert tuple(p[5]) == (7, 1, 1)     # token 5 of a 4-wide frame: row 1, column 1
    assert tuple(p[3]) == (7, 0, 3)
    assert tuple(p[4]) == (7, 1, 0)
    assert tuple(p[15]) == (7, 3, 3)
    # 480p latent frame: 30 rows x 52 columns = 1560 tokens
    p = fo.token_positions([40, 41], 30, 52)
    assert p.shape == (3120, 3)
    assert tuple(p[1559]) == (40, 29, 51)
    assert tuple(p[51]) == (40, 0, 51)
    assert tuple(p[52]) == (40, 1, 0)
    assert tuple(p[1560]) == (41, 0, 0)
    assert tuple(p[1560 + 1559]) == (41, 29, 51)
    # 720p: 45 x 80; a non-square frame catches a swapped (y, x)
    p = fo.token_positions([260], 45, 80)
    assert tuple(p[80 * 44 + 79]) == (260, 44, 79)
    assert tuple(p[81]) == (260, 1, 1)
    # a frame 3 rows x 5 columns, every token by hand
    p = fo.token_positions([0], 3, 5)
    assert [tuple(r[1:]) for r in p] == [(y, x) for y in range(3) for x in range(5)]


def test_attention_rows_is_the_definition_on_the_selected_rows_and_heads():
    # The large GPU tests evaluate the reference on sampled rows (and heads) only;
    # each selected output must equal the pure-Python brute force of that row and head.
    rng = np.random.default_rng(17)
    q = rng.standard_normal((9, 3, 8))
    k = rng.standard_normal((13, 3, 8))
    v = rng.standard_normal((13, 3, 8))
    rows, heads = np.array([0, 4, 8]), np.array([2, 0])
    got = fo.attention_rows_f64(q, k, v, rows, heads)
    assert got.shape == (3, 2, 8)
    for a, r in enumerate(rows):
        for b, hh in enumerate(heads):
            bf = fo.attention_bruteforce([[q[r, hh].tolist()]], [[x.tolist()] for x in k[:, hh]],
                                         [[x.tolist()] for x in v[:, hh]])
            np.testing.assert_allclose(got[a, b], bf[0][0], rtol=0, atol=1e-12)
    # all heads by default
    assert fo.attention_rows_f64(q, k, v, rows).shape == (3, 3, 8)


def test_published_k_is_the_rounded_exact_rotation():
    # Published K = RoPE(K) rounded once to bf16.  Against exact rational arithmetic on
    # the same fp64 cos/sin values (Python's math library, as the contract fixes), each
    # element must be within one bf16 unit in the last place of the exact rotation: a
    # dropped term, a flipped sign or a wrong pairing would be off by far more.
    from fractions import Fraction
    d = 64
    rng = np.random.default_rng(23)
    k = fo.f64_to_bf16_bits(rng.standard_normal((3, 2, d)))
    pos = np.array([[3, 2, 5], [40, 29, 51], [0, 7, 0]], dtype=np.int64)
    got = fo.bf16_bits_to_f64(fo.rope_k_bits(k, pos, d, 10000.0))
    kf = fo.bf16_bits_to_f64(k)
    dt, dy, dx = d - 4 * (d // 6), 2 * (d // 6), 2 * (d // 6)
    axes = [(0, j, dt) for j in range(dt // 2)] + [(1, j, dy) for j in range(dy // 2)] + \
           [(2, j, dx) for j in range(dx // 2)]
    for n in range(3):
        for h in range(2):
            for p, (axis, j, da) in enumerate(axes):
                ang = float(pos[n, axis]) * (10000.0 ** (-(2 * j) / da))
                c, s = Fraction(math.cos(ang)), Fraction(math.sin(ang))
                a, b = Fraction(kf[n, h, 2 * p]), Fraction(kf[n, h, 2 * p + 1])
                for val, exact in ((got[n, h, 2 * p], a * c - b * s), (got[n, h, 2 * p + 1], a * s + b * c)):
                    e = float(exact)
                    ulp = 2.0 ** (math.frexp(e)[1] - 8) if e != 0 else 2.0 ** -133
                    assert abs(val - e) <= ulp, (n, h, p, val, e)
