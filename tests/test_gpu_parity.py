"""Parity of the CUDA path (through the C ABI) against the fp64 oracle.

Bit-exact: Gamma(i), slot tags/frames and published K/V bytes.  Attention
output: max-abs <= 2e-2 and relative L2 <= 5e-3 against the fp64 definition.
"""
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


def _check_stage_slots(bank, obank, layer, stage):
    H = obank.cfg.history
    for s in range(H):
        tag, k, v = bank.slot_tensors(layer, stage, s)
        osl = obank.stage[layer][stage][s]
        assert tag == osl.tag, (stage, s, tag, osl.tag)
        if osl.tag >= 0:
            assert np.array_equal(to_bits(k), osl.k), f"published K differs in slot {s}"
            assert np.array_equal(to_bits(v), osl.v), f"published V differs in slot {s}"


def _check_anchor_slots(bank, obank, layer):
    for s in range(obank.cfg.anchor_capacity):
        tag, k, v = bank.slot_tensors(layer, -1, s)
        osl = obank.anchor[layer][s]
        assert tag == osl.tag
        if osl.tag >= 0:
            assert np.array_equal(to_bits(k), osl.k)
            assert np.array_equal(to_bits(v), osl.v)


def _tiny_run(ff, fields, cfg_id=1):
    from kv_cache_attention_ff_gb300 import synth
    dev = torch.device("cuda:0")
    bank = ff.Bank(**fields)
    ocfg = oracle_cfg(fields)
    obank = fo.OracleBank(ocfg)
    T, h, d = fields["frame_h"] * fields["frame_w"], fields["heads"], fields["head_dim"]
    N, B = fields["total_frames"], fields["chunk_frames"]
    for a0, n in anchor_blocks(fields):
        frames = [a0 + j * fields["anchor_stride"] for j in range(n)]
        kb = synth.frames_tensor(cfg_id, 0, synth.ANCHOR_STREAM, synth.K, frames, T, h, d, "normal")
        vb = synth.frames_tensor(cfg_id, 0, synth.ANCHOR_STREAM, synth.V, frames, T, h, d, "normal")
        bank.anchor_publish(0, a0, n, from_bits(kb, dev), from_bits(vb, dev))
        obank.anchor_publish(0, a0, n, kb, vb)
    _check_anchor_slots(bank, obank, 0)
    worst = (0.0, 0.0)
    for i in range(fo.num_chunks(N, B)):
        s, e = fo.chunk_span(i, B, N)
        frames = list(range(s, e + 1))
        assert bank.gamma(i) == fo.gamma(i, B, fields["anchor_stride"], N)
        for st in range(fields["n_stages"]):
            qb = synth.frames_tensor(cfg_id, 0, st, synth.Q, frames, T, h, d, "normal")
            kb = synth.frames_tensor(cfg_id, 0, st, synth.K, frames, T, h, d, "normal")
            vb = synth.frames_tensor(cfg_id, 0, st, synth.V, frames, T, h, d, "normal")
            out = torch.empty((len(frames) * T, h, d), dtype=torch.bfloat16, device=dev)
            bank.render_attn(0, st, i, from_bits(qb, dev), from_bits(kb, dev), from_bits(vb, dev), out)
            res = obank.render(0, st, i, qb, kb, vb)
            torch.cuda.synchronize()
            mae, rl2, ok = compare_out(out, res.out)
            worst = (max(worst[0], mae), max(worst[1], rl2))
            assert ok, (i, st, mae, rl2)
            _check_stage_slots(bank, obank, 0, st)
    assert bank.error_poll() == 0
    bank.close()
    return worst


def test_tiny_full_schedule(ff):
    fields = CONFIGS["tiny"][1]
    mae, rl2 = _tiny_run(ff, fields)
    assert mae < 2e-2 and rl2 < 5e-3


@pytest.mark.parametrize("H", [1, 3])
def test_tiny_ring_reuse(ff, H):
    # H = 1: every chunk overwrites the slot holding the chunk it attends to.
    fields = dict(CONFIGS["tiny"][1], history=H, n_stages=2)
    _tiny_run(ff, fields, cfg_id=11)


def test_tiny_head_dim_128_odd_frame(ff):
    # d = 128 path on a small ragged case: 5 x 7 tokens per frame, 3 heads.
    fields = dict(CONFIGS["tiny"][1], heads=3, head_dim=128, frame_h=5, frame_w=7, n_stages=1)
    _tiny_run(ff, fields, cfg_id=12)


def test_errors_leave_state_unchanged(ff):
    fields = CONFIGS["tiny"][1]
    dev = torch.device("cuda:0")
    bank = ff.Bank(**fields)
    T, h, d = 16, 2, 64
    z = torch.zeros((3 * T, h, d), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(z)
    with pytest.raises(ff.FFError) as ei:
        bank.render_attn(0, 0, 0, z, z, z, out)
    assert ei.value.code == "FF_ERR_ANCHOR_MISSING"
    z2 = torch.zeros((2 * T, h, d), dtype=torch.bfloat16, device=dev)
    bank.anchor_publish(0, 0, 2, z2, z2)
    with pytest.raises(ff.FFError) as ei:
        bank.render_attn(0, 0, 1, z, z, z, out)
    assert ei.value.code == "FF_ERR_ORDER"
    with pytest.raises(ff.FFError) as ei:
        bank.anchor_publish(0, 2, 1, z2[:T], z2[:T])
    assert ei.value.code == "FF_ERR_ARG"
    with pytest.raises(ff.FFError) as ei:
        bank.render_attn(0, 4, 0, z, z, z, out)
    assert ei.value.code == "FF_ERR_ARG"
    assert bank.slot_info(0, 0, 0)[0] == -1
    bank.render_attn(0, 0, 0, z, z, z, out)
    assert bank.slot_info(0, 0, 0)[:2] == (0, 3)
    with pytest.raises(ff.FFError) as ei:
        bank.render_attn(0, 0, 1, z, z, z, out)   # needs anchor 8
    assert ei.value.code == "FF_ERR_ANCHOR_MISSING"
    assert bank.slot_info(0, 0, 1)[0] == -1
    bank.close()


def test_max_bytes_oom(ff):
    fields = dict(CONFIGS["tiny"][1], max_bytes=1000)
    with pytest.raises(ff.FFError) as ei:
        ff.Bank(**fields)
    assert ei.value.code == "FF_ERR_OOM"


def _big_call(ff, name, check_chunk, full_heads=(0,), n_rows=256, seed=0):
    """Run stage 0 of `name` from chunk 0 to check_chunk; bit-exact slots at every
    chunk, attention on sampled rows (all heads) and full rows for full_heads."""
    from kv_cache_attention_ff_gb300 import synth
    cfg_id, fields, mode = CONFIGS[name]
    fields = dict(fields, n_layers=1)
    dev = torch.device("cuda:0")
    T, h, d = fields["frame_h"] * fields["frame_w"], fields["heads"], fields["head_dim"]
    N, B, D = fields["total_frames"], fields["chunk_frames"], fields["anchor_stride"]
    bank = ff.Bank(**fields)
    ocfg = oracle_cfg(fields)
    obank = fo.OracleBank(ocfg)
    needed_blocks = sorted({a // (3 * D) for i in range(check_chunk + 1) for a in fo.gamma(i, B, D, N)})
    blocks = anchor_blocks(fields)
    for bi in needed_blocks:
        a0, n = blocks[bi]
        frames = [a0 + j * D for j in range(n)]
        kt = synth.device_frames(cfg_id, 0, synth.ANCHOR_STREAM, synth.K, frames, T, h, d, mode)
        vt = synth.device_frames(cfg_id, 0, synth.ANCHOR_STREAM, synth.V, frames, T, h, d, "normal")
        bank.anchor_publish(0, a0, n, kt, vt)
        obank.anchor_publish(0, a0, n, to_bits(kt), to_bits(vt))
    _check_anchor_slots(bank, obank, 0)
    qs = synth.DeviceARStream(cfg_id, 0, 0, synth.Q, T, h, d, mode)
    ks = synth.DeviceARStream(cfg_id, 0, 0, synth.K, T, h, d, mode)
    vs = synth.DeviceARStream(cfg_id, 0, 0, synth.V, T, h, d, "normal")
    rng = np.random.default_rng(seed)
    result = None
    for i in range(check_chunk + 1):
        s, e = fo.chunk_span(i, B, N)
        nf = e - s + 1
        q, k, v = qs.frames(nf), ks.frames(nf), vs.frames(nf)
        out = torch.empty_like(q)
        bank.render_attn(0, 0, i, q, k, v, out)
        qb, kb, vb = to_bits(q), to_bits(k), to_bits(v)
        if i < check_chunk:
            pos = fo.token_positions(list(range(s, e + 1)), fields["frame_h"], fields["frame_w"])
            obank.commit_publish(0, 0, i, fo.rope_k_bits(kb, pos, d, 10000.0), vb)
        else:
            Q, K, V, k_rot = obank.render_context(0, 0, i, qb, kb, vb)
            obank.commit_publish(0, 0, i, k_rot, vb)
            nq = Q.shape[0]
            rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, nq - 73, nq - 1],
                                             rng.choice(nq, n_rows, replace=False)]))
            rows = rows[rows < nq]
            ref = fo.attention_rows_f64(Q, K, V, rows)
            torch.cuda.synchronize()
            got = out[torch.from_numpy(rows).to(dev)]
            mae, rl2, ok = compare_out(got, ref)
            assert ok, ("sampled rows", mae, rl2)
            for hh in full_heads:
                ref_h = fo.attention_f64(Q[:, hh:hh + 1], K[:, hh:hh + 1], V[:, hh:hh + 1])
                mae2, rl22, ok2 = compare_out(out[:, hh:hh + 1], ref_h)
                assert ok2, ("full head", hh, mae2, rl22)
            result = (mae, rl2, K.shape[0])
        torch.cuda.synchronize()
        _check_stage_slots(bank, obank, 0, 0)
    assert bank.error_poll() == 0
    bank.close()
    return result


def test_wan13b_480p_steady_call(ff):
    mae, rl2, nk = _big_call(ff, "wan13b_480p", check_chunk=10)
    assert nk == 31200


def test_wan13b_480p_rampup_chunks(ff):
    # chunk 3: Gamma = (0, 20), 14 key frames; checks a ramp-up (non-steady) key count
    mae, rl2, nk = _big_call(ff, "wan13b_480p", check_chunk=3, full_heads=(), n_rows=128, seed=1)
    assert nk == 14 * 1560


def test_wan14b_480p_steady_call(ff):
    mae, rl2, nk = _big_call(ff, "wan14b_480p", check_chunk=5, full_heads=(39,), n_rows=128, seed=2)
    assert nk == 31200
