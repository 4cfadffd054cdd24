"""Packed block-causal renderer forward on the GPU against the oracle (the
sequential renderer at one stage) and against the library's own sequential calls."""
import numpy as np
import pytest

from oracle import ff_oracle as fo
from tests.ffcases import CONFIGS, compare_out, from_bits, oracle_cfg, to_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ff():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_attention_ff_gb300 import build, ff as ffmod
    build.build()
    return ffmod


@pytest.mark.parametrize("variant", [dict(), dict(history=1), dict(heads=3, head_dim=128, frame_h=5, frame_w=7)])
def test_tiny_packed_matches_oracle(ff, variant):
    from kv_cache_attention_ff_gb300 import synth
    cfg_id, fields, _ = CONFIGS["tiny"]
    fields = dict(fields, n_stages=1, **variant)
    dev = torch.device("cuda:0")
    T, h, d, N = fields["frame_h"] * fields["frame_w"], fields["heads"], fields["head_dim"], 13
    q, k, v = (synth.frames_tensor(cfg_id, 3, 0, t, list(range(N)), T, h, d, "normal") for t in range(3))
    ak = synth.frames_tensor(cfg_id, 3, synth.ANCHOR_STREAM, synth.K, [0, 4, 8, 12], T, h, d, "normal")
    av = synth.frames_tensor(cfg_id, 3, synth.ANCHOR_STREAM, synth.V, [0, 4, 8, 12], T, h, d, "normal")
    bank = ff.Bank(**fields)
    ws = torch.empty(bank.packed_workspace_bytes(), dtype=torch.uint8, device=dev)
    out = torch.empty((N * T, h, d), dtype=torch.bfloat16, device=dev)
    bank.packed_render_attn(*(from_bits(x, dev) for x in (q, k, v, ak, av)), out, ws)
    ref = fo.packed_block_causal(oracle_cfg(fields), q, k, v, ak, av)
    torch.cuda.synchronize()
    mae, rl2, ok = compare_out(out, ref)
    assert ok, (mae, rl2)
    # bank state untouched
    assert all(bank.slot_info(0, 0, s)[0] == -1 for s in range(fields["history"]))
    assert bank.error_poll() == 0
    bank.close()


def test_wan13b_packed_81_latents(ff):
    """One stage of the 81-latent 1.3B 480p clip in one call (27 chunks, 4680 queries
    each, 5..20 key frames); sampled chunks and rows against the oracle, and every
    chunk against the library's sequential ff_render_attn within the same tolerance."""
    from kv_cache_attention_ff_gb300 import synth
    cfg_id, fields, mode = CONFIGS["wan13b_480p"]
    fields = dict(fields, n_stages=1)
    T, h, d, N = 1560, 12, 128, 81
    dev = torch.device("cuda:0")
    q, k = (synth.device_frames(cfg_id, 4, 0, t, list(range(N)), T, h, d, mode) for t in (0, 1))
    v = synth.device_frames(cfg_id, 4, 0, 2, list(range(N)), T, h, d, "normal")
    anchors = list(range(0, 81, 10))
    ak = synth.device_frames(cfg_id, 4, synth.ANCHOR_STREAM, synth.K, anchors, T, h, d, mode)
    av = synth.device_frames(cfg_id, 4, synth.ANCHOR_STREAM, synth.V, anchors, T, h, d, "normal")
    bank = ff.Bank(**fields)
    ws = torch.empty(bank.packed_workspace_bytes(), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    bank.packed_render_attn(q, k, v, ak, av, out, ws)
    # sequential renders through the bank
    for b in range(3):
        sl = slice(3 * b * T, 3 * (b + 1) * T)
        bank.anchor_publish(0, 30 * b, 3, ak[sl].contiguous(), av[sl].contiguous())
    seq = torch.empty_like(q)
    for i in range(27):
        sl = slice(3 * i * T, 3 * (i + 1) * T)
        o = torch.empty((3 * T, h, d), dtype=torch.bfloat16, device=dev)
        bank.render_attn(0, 0, i, q[sl].contiguous(), k[sl].contiguous(), v[sl].contiguous(), o)
        seq[sl] = o
    torch.cuda.synchronize()
    mae, rl2, ok = compare_out(out, seq.to(torch.float64).cpu().numpy())
    assert ok, ("packed vs sequential", mae, rl2)
    # oracle on sampled chunks
    ob = fo.OracleBank(oracle_cfg(fields))
    akb, avb = to_bits(ak), to_bits(av)
    for b in range(3):
        ob.anchor_publish(0, 30 * b, 3, akb[3 * b * T:3 * (b + 1) * T], avb[3 * b * T:3 * (b + 1) * T])
    qb_all, kb_all, vb_all = to_bits(q), to_bits(k), to_bits(v)
    rng = np.random.default_rng(12)
    for i in range(27):
        sl = slice(3 * i * T, 3 * (i + 1) * T)
        qb, kb, vb = qb_all[sl], kb_all[sl], vb_all[sl]
        if i in (0, 3, 13, 26):
            Q, K, V, k_rot = ob.render_context(0, 0, i, qb, kb, vb)
            rows = np.unique(np.concatenate([[0, 4679], rng.choice(4680, 40, replace=False)]))
            ref = fo.attention_rows_f64(Q, K, V, rows)
            got = out[torch.from_numpy(rows + 3 * i * T).to(dev)]
            mae, rl2, ok = compare_out(got, ref)
            assert ok, (i, mae, rl2)
        else:
            k_rot = fo.rope_k_bits(kb, fo.token_positions(list(range(3 * i, 3 * i + 3)), 30, 52), d, 1e4)
        ob.commit_publish(0, 0, i, k_rot, vb)
    assert bank.error_poll() == 0
    bank.close()
