"""Parity on randomly drawn small bank descriptions.

Each seed draws a description (stages, H, B_R, Delta, anchor-ring capacity,
latents, heads, head_dim, frame size) and runs, through the C ABI, against the
fp64 oracle:
  * the whole render schedule (every chunk at every stage), anchors published
    block by block just before the first chunk that needs them, with published
    K/V bytes and slot tags checked bit-exactly after every call;
  * every planner block of a second bank;
  * the packed block-causal forward of one stage;
  * the render schedule of a bank with 1-4 stages issued as stage-wavefront
    batches (ff_render_attn_batch).
The draws cover tokens-per-frame down to 1, short final chunks, anchors inside
chunks, anchor-ring wrap-around and both head sizes, i.e. the segment layouts
the attention kernel reads in place; six larger draws (frames of 20-400 tokens,
up to 8 heads) give segments of many key tiles and split work plans.
"""
import numpy as np
import pytest

from oracle import ff_oracle as fo
from tests.ffcases import compare_out, from_bits, oracle_cfg, to_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SEEDS = list(range(12))
# larger draws (frames of 20-400 tokens, up to 8 heads: segments of many key tiles)
BIG = [100 + s for s in range(6)]


@pytest.fixture(scope="module")
def ff():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_attention_ff_gb300 import build, ff as ffmod
    build.build()
    return ffmod


def _draw(seed):
    if seed >= 100:
        return _draw_big(seed - 100)
    r = np.random.default_rng(1000 + seed)
    B = int(r.integers(1, 5))
    stride = int(r.integers(1, 7))
    N = int(r.integers(5, 25))
    A = fo.num_anchors(N, stride)
    # a ring that holds the anchors of two consecutive 3-anchor blocks plus the
    # widest Gamma(i) span, or every anchor
    need = 3 * (-(-B // stride) + 3)
    cap = A if r.random() < 0.5 else min(A, max(need, 6))
    return dict(n_layers=1, n_stages=int(r.integers(1, 3)), history=int(r.integers(1, 5)), chunk_frames=B,
                anchor_stride=stride, anchor_capacity=cap, total_frames=N, heads=int(r.integers(1, 4)),
                head_dim=int(r.choice([64, 128])), frame_h=int(r.integers(1, 6)), frame_w=int(r.integers(1, 8)))


def _draw_big(seed):
    r = np.random.default_rng(5000 + seed)
    B = int(r.integers(1, 5))
    stride = int(r.integers(2, 9))
    N = int(r.integers(8, 30))
    A = fo.num_anchors(N, stride)
    need = 3 * (-(-B // stride) + 3)
    cap = A if r.random() < 0.5 else min(A, max(need, 6))
    return dict(n_layers=1, n_stages=int(r.integers(1, 3)), history=int(r.integers(1, 6)), chunk_frames=B,
                anchor_stride=stride, anchor_capacity=cap, total_frames=N, heads=int(r.integers(1, 9)),
                head_dim=int(r.choice([64, 128])), frame_h=int(r.integers(4, 21)), frame_w=int(r.integers(5, 21)))


def _check_slots(bank, obank, stage):
    for s in range(obank.cfg.history):
        tag, k, v = bank.slot_tensors(0, stage, s)
        osl = obank.stage[0][stage][s]
        assert tag == osl.tag
        if osl.tag >= 0:
            assert np.array_equal(to_bits(k), osl.k) and np.array_equal(to_bits(v), osl.v)


@pytest.mark.parametrize("seed", SEEDS + BIG)
def test_random_description_render_schedule(ff, seed):
    from kv_cache_attention_ff_gb300 import synth
    f = _draw(seed)
    cfg_id = 200 + seed
    dev = torch.device("cuda:0")
    T, h, d = f["frame_h"] * f["frame_w"], f["heads"], f["head_dim"]
    N, B, S = f["total_frames"], f["chunk_frames"], f["anchor_stride"]
    bank = ff.Bank(**f)
    obank = fo.OracleBank(oracle_cfg(f))
    anchors = list(range(0, N, S))
    published = 0  # anchors published so far (whole 3-anchor blocks, in order)
    for i in range(fo.num_chunks(N, B)):
        g = fo.gamma(i, B, S, N)
        while published < len(anchors) and anchors[published] <= max(g):
            n = min(3, len(anchors) - published)
            frames = anchors[published:published + n]
            kb = synth.frames_tensor(cfg_id, 0, synth.ANCHOR_STREAM, synth.K, frames, T, h, d, "normal")
            vb = synth.frames_tensor(cfg_id, 0, synth.ANCHOR_STREAM, synth.V, frames, T, h, d, "normal")
            bank.anchor_publish(0, frames[0], n, from_bits(kb, dev), from_bits(vb, dev))
            obank.anchor_publish(0, frames[0], n, kb, vb)
            published += n
        s, e = fo.chunk_span(i, B, N)
        frames = list(range(s, e + 1))
        for st in range(f["n_stages"]):
            q, k, v = (synth.frames_tensor(cfg_id, 0, st, t, frames, T, h, d, "normal") for t in range(3))
            out = torch.empty((len(frames) * T, h, d), dtype=torch.bfloat16, device=dev)
            bank.render_attn(0, st, i, from_bits(q, dev), from_bits(k, dev), from_bits(v, dev), out)
            ref = obank.render(0, st, i, q, k, v).out
            torch.cuda.synchronize()
            mae, rl2, ok = compare_out(out, ref)
            assert ok, (f, i, st, mae, rl2)
            _check_slots(bank, obank, st)
    assert bank.error_poll() == 0
    bank.close()


@pytest.mark.parametrize("seed", SEEDS + BIG)
def test_random_description_planner_and_packed(ff, seed):
    from kv_cache_attention_ff_gb300 import synth
    f = _draw(seed)
    r = np.random.default_rng(2000 + seed)
    bp, hp = int(r.integers(1, 4)), int(r.integers(1, 4))
    N, S = f["total_frames"], f["anchor_stride"]
    A = fo.num_anchors(N, S)
    f = dict(f, anchor_capacity=A, planner_block=bp, planner_history=hp, n_stages=1)
    cfg_id = 300 + seed
    dev = torch.device("cuda:0")
    T, h, d = f["frame_h"] * f["frame_w"], f["heads"], f["head_dim"]
    bank = ff.Bank(**f)
    obank = fo.OracleBank(oracle_cfg(f))
    for b in range(fo.num_planner_blocks(N, S, bp)):
        frames = fo.planner_block_anchors(b, bp, S, N)
        q, k, v = (synth.frames_tensor(cfg_id, 0, 60, t, frames, T, h, d, "normal") for t in range(3))
        out = torch.empty((len(frames) * T, h, d), dtype=torch.bfloat16, device=dev)
        bank.planner_attn(0, b, from_bits(q, dev), from_bits(k, dev), from_bits(v, dev), out)
        ref, _ = obank.planner_attn(0, b, q, k, v, planner_block=bp, planner_history=hp)
        torch.cuda.synchronize()
        mae, rl2, ok = compare_out(out, ref)
        assert ok, (f, b, mae, rl2)
        ka = synth.frames_tensor(cfg_id, 0, synth.ANCHOR_STREAM, synth.K, frames, T, h, d, "normal")
        va = synth.frames_tensor(cfg_id, 0, synth.ANCHOR_STREAM, synth.V, frames, T, h, d, "normal")
        bank.anchor_publish(0, frames[0], len(frames), from_bits(ka, dev), from_bits(va, dev))
        obank.anchor_publish(0, frames[0], len(frames), ka, va)
    # packed block-causal forward of one stage over all N frames
    anchors = list(range(0, N, S))
    q, k, v = (synth.frames_tensor(cfg_id, 1, 0, t, list(range(N)), T, h, d, "normal") for t in range(3))
    ak = synth.frames_tensor(cfg_id, 1, synth.ANCHOR_STREAM, synth.K, anchors, T, h, d, "normal")
    av = synth.frames_tensor(cfg_id, 1, synth.ANCHOR_STREAM, synth.V, anchors, T, h, d, "normal")
    ws = torch.empty(bank.packed_workspace_bytes(), dtype=torch.uint8, device=dev)
    out = torch.empty((N * T, h, d), dtype=torch.bfloat16, device=dev)
    bank.packed_render_attn(*(from_bits(x, dev) for x in (q, k, v, ak, av)), out, ws)
    ref = fo.packed_block_causal(oracle_cfg(f), q, k, v, ak, av)
    torch.cuda.synchronize()
    mae, rl2, ok = compare_out(out, ref)
    assert ok, (f, "packed", mae, rl2)
    assert bank.error_poll() == 0
    bank.close()


@pytest.mark.parametrize("seed", SEEDS + BIG)
def test_random_description_wavefront_batches(ff, seed):
    """The render schedule of a drawn description with 1-4 stages issued as
    stage-wavefront batches (ff_render_attn_batch: at step w, stage k renders
    chunk w - k), every anchor resident; each call against the oracle, slot
    bytes after every batch."""
    from kv_cache_attention_ff_gb300 import synth
    r = np.random.default_rng(3000 + seed)
    f = _draw(seed)
    N, B, S = f["total_frames"], f["chunk_frames"], f["anchor_stride"]
    f = dict(f, n_stages=int(r.integers(1, 5)), anchor_capacity=fo.num_anchors(N, S))
    cfg_id = 400 + seed
    dev = torch.device("cuda:0")
    T, h, d = f["frame_h"] * f["frame_w"], f["heads"], f["head_dim"]
    bank = ff.Bank(**f)
    obank = fo.OracleBank(oracle_cfg(f))
    anchors = list(range(0, N, S))
    kb = synth.frames_tensor(cfg_id, 0, synth.ANCHOR_STREAM, synth.K, anchors, T, h, d, "normal")
    vb = synth.frames_tensor(cfg_id, 0, synth.ANCHOR_STREAM, synth.V, anchors, T, h, d, "normal")
    for j in range(0, len(anchors), 3):
        n = min(3, len(anchors) - j)
        sl = slice(j * T, (j + n) * T)
        bank.anchor_publish(0, anchors[j], n, from_bits(kb[sl], dev), from_bits(vb[sl], dev))
        obank.anchor_publish(0, anchors[j], n, kb[sl], vb[sl])
    nc, ns = fo.num_chunks(N, B), f["n_stages"]
    for w in range(nc + ns - 1):
        calls, refs = [], []
        for st in range(ns):
            i = w - st
            if not 0 <= i < nc:
                continue
            s, e = fo.chunk_span(i, B, N)
            frames = list(range(s, e + 1))
            q, k, v = (synth.frames_tensor(cfg_id, 0, st, t, frames, T, h, d, "normal") for t in range(3))
            out = torch.full((len(frames) * T, h, d), float("nan"), dtype=torch.bfloat16, device=dev)
            calls.append((0, st, i, from_bits(q, dev), from_bits(k, dev), from_bits(v, dev), out))
            refs.append(obank.render(0, st, i, q, k, v).out)
        bank.render_attn_batch(calls)
        torch.cuda.synchronize()
        for c, ref in zip(calls, refs):
            mae, rl2, ok = compare_out(c[6], ref)
            assert ok, (f, w, c[1], c[2], mae, rl2)
            _check_slots(bank, obank, c[1])
    assert bank.error_poll() == 0
    bank.close()
