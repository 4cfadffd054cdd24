"""Parity of ff_render_attn_batch, the stage-wavefront form of the renderer call
(FlashForward, onedev.kr/papers/332, "어떻게 동작하나": the S denoising stages
work on different in-flight chunks at once, stage k on chunk w - k at wavefront
step w).  A batch must give each call's result and bank state exactly as
ff_render_attn would: published K/V bytes and slot tags bit-exact against the
fp64 oracle after every batch, attention within max-abs 2e-2 / rel-L2 5e-3."""
import ctypes

import numpy as np
import pytest

from oracle import ff_oracle as fo
from tests.ffcases import CONFIGS, anchor_blocks, compare_out, from_bits, oracle_cfg, to_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ff():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_attention_ff_gb300 import build, ff as ffmod
    build.build()
    return ffmod


def _publish_all_anchors(bank, obank, fields, cfg_id, dev):
    from kv_cache_attention_ff_gb300 import synth
    T, h, d = fields["frame_h"] * fields["frame_w"], fields["heads"], fields["head_dim"]
    for a0, n in anchor_blocks(fields):
        frames = [a0 + j * fields["anchor_stride"] for j in range(n)]
        kb = synth.frames_tensor(cfg_id, 0, synth.ANCHOR_STREAM, synth.K, frames, T, h, d, "normal")
        vb = synth.frames_tensor(cfg_id, 0, synth.ANCHOR_STREAM, synth.V, frames, T, h, d, "normal")
        bank.anchor_publish(0, a0, n, from_bits(kb, dev), from_bits(vb, dev))
        obank.anchor_publish(0, a0, n, kb, vb)


def _check_slots(bank, obank, stage):
    for s in range(obank.cfg.history):
        tag, k, v = bank.slot_tensors(0, stage, s)
        osl = obank.stage[0][stage][s]
        assert tag == osl.tag, (stage, s, tag, osl.tag)
        if osl.tag >= 0:
            assert np.array_equal(to_bits(k), osl.k) and np.array_equal(to_bits(v), osl.v), (stage, s)


def _wavefront(fields, same_chunk):
    """Batches of one wavefront step each: stage k renders chunk w - k (or, with
    same_chunk, every stage renders chunk w)."""
    S, nc = fields["n_stages"], fo.num_chunks(fields["total_frames"], fields["chunk_frames"])
    steps = []
    for w in range(nc + (0 if same_chunk else S - 1)):
        calls = [(k, w if same_chunk else w - k) for k in range(S)]
        steps.append([(k, i) for k, i in calls if 0 <= i < nc])
    return steps


@pytest.mark.parametrize("same_chunk", [False, True])
@pytest.mark.parametrize("variant", ["tiny", "tiny_h1_d128"])
def test_tiny_wavefront_batches_match_oracle(ff, variant, same_chunk):
    from kv_cache_attention_ff_gb300 import synth
    fields = dict(CONFIGS["tiny"][1])
    if variant == "tiny_h1_d128":
        fields.update(history=1, heads=3, head_dim=128, frame_h=5, frame_w=7)
    cfg_id = 21
    dev = torch.device("cuda:0")
    bank = ff.Bank(**fields)
    obank = fo.OracleBank(oracle_cfg(fields))
    _publish_all_anchors(bank, obank, fields, cfg_id, dev)
    T, h, d = fields["frame_h"] * fields["frame_w"], fields["heads"], fields["head_dim"]
    N, B = fields["total_frames"], fields["chunk_frames"]
    bank.set_timing(True)
    n_calls = 0
    for step in _wavefront(fields, same_chunk):
        calls, refs = [], []
        for st, i in step:
            s, e = fo.chunk_span(i, B, N)
            frames = list(range(s, e + 1))
            qb, kb, vb = (synth.frames_tensor(cfg_id, 0, st, t, frames, T, h, d, "normal") for t in (0, 1, 2))
            out = torch.full((len(frames) * T, h, d), float("nan"), dtype=torch.bfloat16, device=dev)
            calls.append((0, st, i, from_bits(qb, dev), from_bits(kb, dev), from_bits(vb, dev), out))
            refs.append(obank.render(0, st, i, qb, kb, vb).out)
        bank.render_attn_batch(calls)
        n_calls += len(calls)
        torch.cuda.synchronize()
        for (layer, st, i, q, k, v, out), ref in zip(calls, refs):
            mae, rl2, ok = compare_out(out, ref)
            assert ok, (variant, st, i, mae, rl2)
            _check_slots(bank, obank, st)
    t = bank.read_timing()
    assert t.calls == n_calls and t.launches >= 2 * len(_wavefront(fields, same_chunk))
    bank.set_timing(False)
    assert bank.error_poll() == 0
    bank.close()


def test_batch_errors_leave_state_unchanged(ff):
    fields = dict(CONFIGS["tiny"][1])
    dev = torch.device("cuda:0")
    bank = ff.Bank(**fields)
    T, h, d = 16, 2, 64
    z = torch.zeros((3 * T, h, d), dtype=torch.bfloat16, device=dev)
    z4 = torch.zeros((4 * T, h, d), dtype=torch.bfloat16, device=dev)
    bank.anchor_publish(0, 0, 4, z4, z4)
    outs = [torch.full_like(z, 7.0) for _ in range(4)]
    # a repeated stage
    with pytest.raises(ff.FFError) as ei:
        bank.render_attn_batch([(0, 1, 0, z, z, z, outs[0]), (0, 1, 0, z, z, z, outs[1])])
    assert ei.value.code == "FF_ERR_ARG"
    # the last call out of order: nothing of the batch runs
    with pytest.raises(ff.FFError) as ei:
        bank.render_attn_batch([(0, 0, 0, z, z, z, outs[0]), (0, 1, 0, z, z, z, outs[1]), (0, 2, 1, z, z, z, outs[2])])
    assert ei.value.code == "FF_ERR_ORDER"
    # too many calls, or none
    lib = ff.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    arr = (ff.RenderCall * 5)()
    assert ff.STATUS[lib.ff_render_attn_batch(bank.handle, 5, arr, stream)] == "FF_ERR_ARG"
    assert ff.STATUS[lib.ff_render_attn_batch(bank.handle, 0, arr, stream)] == "FF_ERR_ARG"
    torch.cuda.synchronize()
    assert all(bool((o == 7.0).all()) for o in outs)
    for st in range(4):
        assert [bank.slot_info(0, st, s)[0] for s in range(2)] == [-1, -1]
    # the same calls in order now run
    bank.render_attn_batch([(0, 0, 0, z, z, z, outs[0]), (0, 1, 0, z, z, z, outs[1]), (0, 2, 0, z, z, z, outs[2])])
    torch.cuda.synchronize()
    assert [bank.slot_info(0, st, 0)[0] for st in range(4)] == [0, 0, 0, -1]
    assert bank.error_poll() == 0
    bank.close()


def test_wan13b_480p_four_stage_batch_sampled(ff):
    """The 1.3B 480p steady call at all four stages in one batch (chunk 5 of each
    stage after batches of chunks 0..4): slot bytes bit-exact, sampled rows of every
    call against the oracle's context."""
    from kv_cache_attention_ff_gb300 import synth
    cfg_id, fields, mode = CONFIGS["wan13b_480p"]
    T, h, d = 1560, fields["heads"], fields["head_dim"]
    dev = torch.device("cuda:0")
    bank = ff.Bank(**fields)
    ob = fo.OracleBank(oracle_cfg(fields))
    ka = synth.device_frames(cfg_id, 0, synth.ANCHOR_STREAM, synth.K, [0, 10, 20], T, h, d, mode)
    va = synth.device_frames(cfg_id, 0, synth.ANCHOR_STREAM, synth.V, [0, 10, 20], T, h, d, "normal")
    bank.anchor_publish(0, 0, 3, ka, va)
    ob.anchor_publish(0, 0, 3, to_bits(ka), to_bits(va))
    streams = {st: [synth.DeviceARStream(cfg_id, 0, st, t, T, h, d, mode if t < 2 else "normal")
                    for t in (synth.Q, synth.K, synth.V)] for st in range(4)}
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, 4607, 4608, 4679], rng.choice(4680, 40, replace=False)]))
    outs = [torch.empty((3 * T, h, d), dtype=torch.bfloat16, device=dev) for _ in range(4)]
    for i in range(6):
        s, e = fo.chunk_span(i, 3, 81)
        pos = fo.token_positions(list(range(s, e + 1)), 30, 52)
        inputs = [[x.frames(3) for x in streams[st]] for st in range(4)]
        bank.render_attn_batch([(0, st, i, *inputs[st], outs[st]) for st in range(4)])
        torch.cuda.synchronize()
        for st in range(4):
            qb, kb, vb = (to_bits(x) for x in inputs[st])
            if i == 5:
                Q, K, V, k_rot = ob.render_context(0, st, i, qb, kb, vb)
                ref = fo.attention_rows_f64(Q, K, V, rows)
                mae, rl2, ok = compare_out(outs[st][torch.from_numpy(rows).to(dev)], ref)
                assert ok, (st, mae, rl2)
            else:
                k_rot = fo.rope_k_bits(kb, pos, d, 10000.0)
            ob.commit_publish(0, st, i, k_rot, vb)
            tag, sk, sv = bank.slot_tensors(0, st, i % 5)
            assert tag == i and np.array_equal(to_bits(sk), k_rot) and np.array_equal(to_bits(sv), vb), (st, i)
    assert bank.error_poll() == 0
    bank.close()


def test_wan14b_480p_four_stage_batch_sampled_heads(ff):
    """The 14B 480p shape (40 heads, 4680 queries over 31200 keys) at all four stages
    in one batch (chunk 5 of each stage after batches of chunks 0..4): slot bytes
    bit-exact on 3 heads at every chunk, sampled rows of 3 heads of every call
    against the oracle's definition on those heads."""
    from kv_cache_attention_ff_gb300 import synth
    cfg_id, fields, mode = CONFIGS["wan14b_480p"]
    T, h, d = 1560, fields["heads"], fields["head_dim"]
    dev = torch.device("cuda:0")
    heads = np.array([0, 21, 39])
    bank = ff.Bank(**fields)
    ka = synth.device_frames(cfg_id, 0, synth.ANCHOR_STREAM, synth.K, [0, 10, 20], T, h, d, mode)
    va = synth.device_frames(cfg_id, 0, synth.ANCHOR_STREAM, synth.V, [0, 10, 20], T, h, d, "normal")
    bank.anchor_publish(0, 0, 3, ka, va)
    anc_k = {a: fo.rope_k_bits(to_bits(ka[j * T:(j + 1) * T])[:, heads], fo.token_positions([a], 30, 52), d, 1e4)
             for j, a in enumerate((0, 10, 20))}
    anc_v = {a: to_bits(va[j * T:(j + 1) * T])[:, heads] for j, a in enumerate((0, 10, 20))}
    streams = {st: [synth.DeviceARStream(cfg_id, 0, st, t, T, h, d, mode if t < 2 else "normal")
                    for t in (synth.Q, synth.K, synth.V)] for st in range(4)}
    hist = {st: {} for st in range(4)}   # chunk -> (rotated K bits, V bits) of the checked heads
    rng = np.random.default_rng(13)
    rows = np.unique(np.concatenate([[0, 255, 256, 4607, 4608, 4679], rng.choice(4680, 26, replace=False)]))
    outs = [torch.empty((3 * T, h, d), dtype=torch.bfloat16, device=dev) for _ in range(4)]
    for i in range(6):
        s, e = fo.chunk_span(i, 3, 81)
        pos = fo.token_positions(list(range(s, e + 1)), 30, 52)
        inputs = [[x.frames(3) for x in streams[st]] for st in range(4)]
        bank.render_attn_batch([(0, st, i, *inputs[st], outs[st]) for st in range(4)])
        torch.cuda.synchronize()
        for st in range(4):
            q, k, v = (to_bits(x)[:, heads] for x in inputs[st])
            k_rot = fo.rope_k_bits(k, pos, d, 1e4)
            hist[st][i] = (k_rot, v)
            tag, sk, sv = bank.slot_tensors(0, st, i % 5)
            assert tag == i
            assert np.array_equal(to_bits(sk)[:, heads], k_rot) and np.array_equal(to_bits(sv)[:, heads], v), (st, i)
            if i == 5:
                ks = [anc_k[a] for a in (10, 20)] + [hist[st][j][0] for j in range(0, 6)]
                vs = [anc_v[a] for a in (10, 20)] + [hist[st][j][1] for j in range(0, 6)]
                K = fo.bf16_bits_to_f64(np.concatenate(ks))
                V = fo.bf16_bits_to_f64(np.concatenate(vs))
                assert K.shape[0] == 20 * T
                Q = fo.rope_q_f64(q, pos, d, 1e4)
                ref = fo.attention_rows_f64(Q, K, V, rows)
                got = outs[st][torch.from_numpy(rows).to(dev)][:, torch.from_numpy(heads).to(dev)]
                mae, rl2, ok = compare_out(got, ref)
                assert ok, (st, mae, rl2)
    assert bank.error_poll() == 0
    bank.close()
