"""CPU-side checks of libff: it loads, exports every entry point that
include/ff.h declares, and its host-only chunk planner agrees with the
oracle's schedule."""
import ctypes
import os
import re

import pytest

from oracle import ff_oracle as fo

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ff():
    from kv_cache_attention_ff_gb300 import build, ff as ffmod
    build.build()
    return ffmod


def _declared():
    src = open(os.path.join(ROOT, "include", "ff.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(ff_\w+)\s*\(", src, re.M)))


def test_exports_every_declared_symbol(ff):
    names = _declared()
    assert "ff_render_attn" in names and "ff_bank_create" in names
    lib = ctypes.CDLL(ff.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(ff.EXPORTS) == names


def test_status_strings(ff):
    for code in range(8):
        assert ff.lib().ff_status_string(code)
    assert ff.lib().ff_status_string(2) == b"chunk out of order for this (layer, stage)"


@pytest.mark.parametrize("fields", [
    dict(total_frames=81, chunk_frames=3, anchor_stride=10, history=5),
    dict(total_frames=13, chunk_frames=3, anchor_stride=4, history=2, anchor_capacity=4, heads=2, head_dim=64,
         frame_h=4, frame_w=4),
    dict(total_frames=261, chunk_frames=3, anchor_stride=10, history=5, anchor_capacity=6),
    dict(total_frames=75, chunk_frames=3, anchor_stride=10, history=1),
    dict(total_frames=50, chunk_frames=4, anchor_stride=7, history=3),
])
def test_plan_matches_oracle(ff, fields):
    d = ff.make_desc(**fields)
    N, B, S, H = fields["total_frames"], fields["chunk_frames"], fields["anchor_stride"], fields["history"]
    for i in range(fo.num_chunks(N, B)):
        p = ff.plan_chunk(d, i)
        s, e = fo.chunk_span(i, B, N)
        g = fo.gamma(i, B, S, N)
        hist = fo.history_chunks(i, H)
        assert (p.first_frame, p.n_frames) == (s, e - s + 1)
        assert list(p.anchors)[:p.n_anchors] == g and p.n_anchors == len(g)
        assert p.n_hist == len(hist) and (not hist or p.hist_first == hist[0])
        hf = sum(fo.chunk_span(j, B, N)[1] - fo.chunk_span(j, B, N)[0] + 1 for j in hist)
        assert p.hist_frames == hf
        assert p.slot == fo.bank_slot(i, H)
        assert p.key_frames == len(g) + hf + (e - s + 1)
    with pytest.raises(ff.FFError) as ei:
        ff.plan_chunk(d, fo.num_chunks(N, B))
    assert ei.value.code == "FF_ERR_ARG"


def test_invalid_descriptions_rejected_before_device(ff):
    for bad in (dict(head_dim=96), dict(history=0), dict(chunk_frames=0), dict(heads=0), dict(rope_theta=0.0),
                dict(history=60)):
        d = ff.make_desc(**bad)
        h = ctypes.c_void_p()
        assert ff.lib().ff_bank_create(ctypes.byref(d), ctypes.byref(h)) == 1
        assert not h.value


def test_create_without_gpu_fails_cleanly(ff):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    d = ff.make_desc()
    h = ctypes.c_void_p()
    assert ff.lib().ff_bank_create(ctypes.byref(d), ctypes.byref(h)) in (5, 7)
    assert not h.value
    assert ff.lib().ff_bank_destroy(None) == 0


def test_synth_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    import numpy as np
    from kv_cache_attention_ff_gb300 import synth
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 3
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.f32_to_bf16_bits(x), ref)
    got = synth._bf16_torch(torch.from_numpy(x)).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("fields", [
    dict(total_frames=81, anchor_stride=10, planner_block=3, planner_history=6),
    dict(total_frames=261, anchor_stride=10, planner_block=3, planner_history=6, anchor_capacity=27),
    dict(total_frames=13, anchor_stride=4, planner_block=3, planner_history=1, anchor_capacity=4),
    dict(total_frames=100, anchor_stride=7, planner_block=2, planner_history=3),
])
def test_planner_plan_matches_oracle(ff, fields):
    d = ff.make_desc(**fields)
    N, S, B, H = fields["total_frames"], fields["anchor_stride"], fields["planner_block"], fields["planner_history"]
    nb = fo.num_planner_blocks(N, S, B)
    for b in range(nb):
        p = ff.plan_planner_block(d, b)
        own = fo.planner_block_anchors(b, B, S, N)
        hist = fo.planner_history_blocks(b, H)
        assert p.first_anchor * S == own[0] and p.n_anchors == len(own)
        assert p.n_hist_blocks == len(hist) and (not hist or p.hist_first_block == hist[0])
        assert p.key_frames == len(own) + B * len(hist)
    with pytest.raises(ff.FFError):
        ff.plan_planner_block(d, nb)


def test_entry_points_reject_a_null_bank(ff):
    # Every entry point that takes a bank returns FF_ERR_ARG for a null one, on the
    # host, before any device work (no GPU needed).
    lib = ff.lib()
    null = ctypes.c_void_p()
    p = ctypes.c_void_p(16)  # never dereferenced: the bank check comes first
    assert lib.ff_anchor_publish(null, 0, 0, 1, p, p, None) == 1
    assert lib.ff_render_attn(null, 0, 0, 0, p, p, p, p, None) == 1
    calls = (ff.RenderCall * 2)()
    assert lib.ff_render_attn_batch(null, 2, calls, None) == 1
    assert lib.ff_planner_attn(null, 0, 0, p, p, p, p, None) == 1
    n = ctypes.c_size_t()
    assert lib.ff_packed_workspace_bytes(null, ctypes.byref(n)) == 1
    assert lib.ff_bank_bytes(null, ctypes.byref(n)) == 1
    assert lib.ff_bank_error_poll(null) == 1
    assert lib.ff_bank_set_timing(null, 1) == 1
    t = ff.KernelTimes()
    assert lib.ff_bank_read_timing(null, ctypes.byref(t)) == 1
    c = ctypes.c_int()
    assert lib.ff_render_kernel_count(null, 0, ctypes.byref(c)) == 1
    assert lib.ff_bank_wait_probe(null, 10, None) == 1
    assert lib.ff_bank_destroy(null) == 0


def test_noalloc_rejects_bad_arguments_on_the_host(ff):
    # Null pointers, unsupported head sizes, misaligned pointers and sizes past the
    # index limits are refused before the library touches a device.
    lib = ff.lib()
    p = ctypes.c_void_p(256)
    odd = ctypes.c_void_p(258)
    assert lib.ff_attention_noalloc(None, p, p, p, 16, 16, 1, 64, None) == 1
    assert lib.ff_attention_noalloc(p, p, p, p, 16, 16, 1, 96, None) == 1
    assert lib.ff_attention_noalloc(p, odd, p, p, 16, 16, 1, 64, None) == 1
    assert lib.ff_attention_noalloc(p, p, p, p, 16, 1 << 25, 1, 64, None) == 1
    assert lib.ff_attention_noalloc(p, p, p, p, 0, 16, 1, 64, None) == 1
