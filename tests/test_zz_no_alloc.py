"""ff_attention_noalloc: attention for callers that cannot allocate device memory.

Some callers cannot let a library call cudaMalloc: code recorded into a CUDA
stream capture (allocation is not a capturable operation), hosts whose device
memory belongs to another caching allocator, processes that must not grow
their footprint after start-up.  ff_attention_noalloc keeps its split
scratch in one fixed static device array instead.  These tests call it through
the C ABI and check, on two calls in a row each:

* the 1.3B 480p renderer call (4680 queries over 31200 keys, 12 heads): the
  output matches the fp64 oracle on the oracle's own rotated queries and
  context, and matches ff_render_attn's output for the same chunk within the
  attention tolerance of the parity tests;
* the 14B 480p shape (40 heads), which runs as whole units with no partials:
  accepted, and sampled rows match the oracle;
* a context of at most one key tile (no split);
* sizes beyond the kernels' index limits are refused before any work.

Collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.
"""
import ctypes

import numpy as np
import pytest

from oracle import ff_oracle as fo
from tests.ffcases import CONFIGS, compare_out, from_bits, oracle_cfg, to_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROWS = np.array([0, 1, 127, 128, 255, 256, 1000, 2047, 3333, 4095, 4607, 4608, 4679])


@pytest.fixture(scope="module")
def ff():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_attention_ff_gb300 import build, ff as ffmod
    build.build()
    return ffmod


def _twice(ff, q, k, v):
    outs = []
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        ff.attention_noalloc(q, k, v, out)
        torch.cuda.synchronize()
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    return outs


def test_noalloc_13b_call_matches_oracle_and_render_attn(ff):
    from kv_cache_attention_ff_gb300 import synth
    cfg_id, fields, mode = CONFIGS["wan13b_480p"]
    fields = dict(fields, n_stages=1)
    dev = torch.device("cuda:0")
    T, h, d = 1560, fields["heads"], fields["head_dim"]
    # oracle side: anchors 0, 10, 20, chunks 0..4 published, then chunk 5
    # (frames 15..17, Gamma = (10, 20)): its rotated Q and context [A_10; A_20; chunks 0..4; own]
    ob = fo.OracleBank(oracle_cfg(fields))
    ka = synth.frames_tensor(cfg_id, 0, synth.ANCHOR_STREAM, synth.K, [0, 10, 20], T, h, d, mode)
    va = synth.frames_tensor(cfg_id, 0, synth.ANCHOR_STREAM, synth.V, [0, 10, 20], T, h, d, "normal")
    ob.anchor_publish(0, 0, 3, ka, va)
    frames = list(range(18))
    qa = synth.frames_tensor(cfg_id, 0, 0, synth.Q, frames, T, h, d, mode)
    kk = synth.frames_tensor(cfg_id, 0, 0, synth.K, frames, T, h, d, mode)
    vv = synth.frames_tensor(cfg_id, 0, 0, synth.V, frames, T, h, d, "normal")
    sl = lambda x, i: x[3 * i * T:3 * (i + 1) * T]
    for i in range(5):
        _, _, _, k_rot = ob.render_context(0, 0, i, sl(qa, i), sl(kk, i), sl(vv, i))
        ob.commit_publish(0, 0, i, k_rot, sl(vv, i))
    Q, K, V, _ = ob.render_context(0, 0, 5, sl(qa, 5), sl(kk, 5), sl(vv, 5))
    assert K.shape[0] == 20 * T
    q_rot = from_bits(fo.f64_to_bf16_bits(Q), dev)
    kc = from_bits(fo.f64_to_bf16_bits(K), dev)   # exact: K, V hold bf16 values
    vc = from_bits(fo.f64_to_bf16_bits(V), dev)
    outs = _twice(ff, q_rot, kc, vc)
    # the definition on exactly the inputs of the call, sampled rows, all heads
    ref_rows = fo.attention_rows_f64(fo.bf16_bits_to_f64(to_bits(q_rot)), K, V, ROWS)
    for out in outs:
        mae, rl2, ok = compare_out(out[ROWS], ref_rows)
        assert ok, (mae, rl2)

    # the existing entry point on the same chunk: ff_render_attn of chunk 5 after chunks 0..4
    bank = ff.Bank(**fields)
    bank.anchor_publish(0, 0, 3, from_bits(ka, dev), from_bits(va, dev))
    ref = None
    for i in range(6):
        q, k, v = (from_bits(sl(x, i), dev) for x in (qa, kk, vv))
        ref = torch.empty_like(q)
        bank.render_attn(0, 0, i, q, k, v, ref)
    torch.cuda.synchronize()
    assert bank.error_poll() == 0
    ref64 = ref.to(torch.float64).cpu().numpy()
    for out in outs:
        mae, rl2, ok = compare_out(out, ref64)
        assert ok, (mae, rl2)
    bank.close()


def test_noalloc_14b_480p_runs_whole_units(ff):
    # 40 heads x 19 query blocks = 760 units: 5 whole waves on 152 SMs, no partials
    from kv_cache_attention_ff_gb300 import synth
    dev = torch.device("cuda:0")
    T, h, d = 1560, 40, 128
    q = synth.device_frames(4, 0, 0, synth.Q, [15, 16, 17], T, h, d, "ar")
    k = synth.device_frames(4, 0, 0, synth.K, list(range(20)), T, h, d, "ar")
    v = synth.device_frames(4, 0, 0, synth.V, list(range(20)), T, h, d, "normal")
    outs = _twice(ff, q, k, v)
    heads = np.array([0, 17, 39])
    qh = fo.bf16_bits_to_f64(to_bits(q[:, heads]))
    kh = fo.bf16_bits_to_f64(to_bits(k[:, heads]))
    vh = fo.bf16_bits_to_f64(to_bits(v[:, heads]))
    ref = fo.attention_rows_f64(qh, kh, vh, ROWS)
    for out in outs:
        mae, rl2, ok = compare_out(out[ROWS][:, heads], ref)
        assert ok, (mae, rl2)


def test_noalloc_single_key_tile(ff):
    # at most 128 keys: one key tile, nothing to split; ragged query and key counts
    rng = np.random.default_rng(7)
    dev = torch.device("cuda:0")
    for nq, nk, h, d in ((300, 100, 3, 64), (37, 128, 2, 128), (1, 1, 1, 64)):
        qb = fo.f64_to_bf16_bits(rng.standard_normal((nq, h, d)))
        kb = fo.f64_to_bf16_bits(rng.standard_normal((nk, h, d)))
        vb = fo.f64_to_bf16_bits(rng.standard_normal((nk, h, d)))
        outs = _twice(ff, from_bits(qb, dev), from_bits(kb, dev), from_bits(vb, dev))
        ref = fo.attention_f64(fo.bf16_bits_to_f64(qb), fo.bf16_bits_to_f64(kb), fo.bf16_bits_to_f64(vb))
        for out in outs:
            mae, rl2, ok = compare_out(out, ref)
            assert ok, (nq, nk, h, d, mae, rl2)


def test_noalloc_refuses_sizes_beyond_index_limits(ff):
    # nk * heads * head_dim >= 2^31 is refused on the host before any pointer is used
    dev = torch.device("cuda:0")
    q = torch.zeros((256, 1, 64), dtype=torch.bfloat16, device=dev)
    out = torch.zeros_like(q)
    lib = ff.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.ff_attention_noalloc(p(q), p(q), p(q), p(out), 256, 1 << 25, 1, 64, stream)
    assert ff.STATUS[rc] == "FF_ERR_ARG"
    rc = lib.ff_attention_noalloc(p(q), p(q), p(q), p(out), 256, 256, 1, 96, stream)   # head_dim 96
    assert ff.STATUS[rc] == "FF_ERR_ARG"
    torch.cuda.synchronize()
    assert int(out.abs().sum()) == 0
