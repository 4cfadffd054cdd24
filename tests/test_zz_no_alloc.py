"""ff_attention_noalloc: attention for callers that cannot allocate device memory.

Callers inside a stream capture, or under a host allocator that owns the
device memory, cannot let the library call cudaMalloc; this entry point keeps
its split scratch in a fixed static device array instead.  The test checks,
through the C ABI, that two calls in a row give the same attention output as
ff_render_attn on the same context (within the attention tolerance of the
parity tests), and that a problem larger than the static scratch is refused.
Collected last on purpose: a failure here does not hide the other GPU tests.
"""
import numpy as np
import pytest

from oracle import ff_oracle as fo
from tests.ffcases import CONFIGS, compare_out, from_bits, to_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ff():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_attention_ff_gb300 import build, ff as ffmod
    build.build()
    return ffmod


def test_noalloc_matches_render_attn_twice(ff):
    from kv_cache_attention_ff_gb300 import synth
    cfg_id, fields, mode = CONFIGS["wan13b_480p"]
    fields = dict(fields, n_stages=1)
    dev = torch.device("cuda:0")
    T, h, d = 1560, fields["heads"], fields["head_dim"]
    bank = ff.Bank(**fields)
    frames = [0, 10, 20]
    ka = synth.device_frames(cfg_id, 0, synth.ANCHOR_STREAM, synth.K, frames, T, h, d, mode)
    va = synth.device_frames(cfg_id, 0, synth.ANCHOR_STREAM, synth.V, frames, T, h, d, "normal")
    bank.anchor_publish(0, 0, 3, ka, va)
    qs = synth.DeviceARStream(cfg_id, 0, 0, synth.Q, T, h, d, mode)
    ks = synth.DeviceARStream(cfg_id, 0, 0, synth.K, T, h, d, mode)
    vs = synth.DeviceARStream(cfg_id, 0, 0, synth.V, T, h, d, "normal")
    for i in range(5):
        q, k, v = qs.frames(3), ks.frames(3), vs.frames(3)
        bank.render_attn(0, 0, i, q, k, v, torch.empty_like(q))
    torch.cuda.synchronize()
    _, k0, v0 = bank.slot_tensors(0, 0, 0)           # chunk 0: overwritten by chunk 5 below
    k0, v0 = k0.clone(), v0.clone()
    q, k, v = qs.frames(3), ks.frames(3), vs.frames(3)
    ref = torch.empty_like(q)
    bank.render_attn(0, 0, 5, q, k, v, ref)          # chunk 5 = frames 15..17, Gamma = (10, 20)
    torch.cuda.synchronize()
    parts_k, parts_v = [], []
    for a in (10, 20):
        _, ak, av = bank.slot_tensors(0, -1, a // 10)
        parts_k.append(ak)
        parts_v.append(av)
    parts_k.append(k0)
    parts_v.append(v0)
    for c in (1, 2, 3, 4, 5):
        _, sk, sv = bank.slot_tensors(0, 0, c % 5)
        parts_k.append(sk)
        parts_v.append(sv)
    kc = torch.cat(parts_k).view(torch.bfloat16).contiguous()
    vc = torch.cat(parts_v).view(torch.bfloat16).contiguous()
    assert kc.shape[0] == 20 * T
    pos = fo.token_positions([15, 16, 17], 30, 52)
    q_rot = from_bits(fo.f64_to_bf16_bits(fo.rope_q_f64(to_bits(q), pos, d, 10000.0)), dev)
    ref64 = ref.to(torch.float64).cpu().numpy()
    outs = []
    for _ in range(2):
        out = torch.full_like(q_rot, float("nan"))
        ff.attention_noalloc(q_rot, kc, vc, out)
        torch.cuda.synchronize()
        mae, rl2, ok = compare_out(out, ref64)
        assert ok, (mae, rl2)
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    bank.close()


def test_noalloc_rejects_problem_beyond_static_scratch(ff):
    dev = torch.device("cuda:0")
    q = torch.zeros((4680, 40, 128), dtype=torch.bfloat16, device=dev)
    k = torch.zeros((256, 40, 128), dtype=torch.bfloat16, device=dev)
    out = torch.zeros_like(q)
    with pytest.raises(ff.FFError) as ei:
        ff.attention_noalloc(q, k, k, out)
    assert ei.value.code == "FF_ERR_ARG"
    torch.cuda.synchronize()
    assert int(out.abs().sum()) == 0
