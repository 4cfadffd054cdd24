"""Planner-role attention on the GPU against the oracle: each planner block attends
block-causally over the clean anchor KV of the previous H_P blocks plus itself
(onedev.kr/papers/332, "무엇과 다른가" and "어떻게 쓰나")."""
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


@pytest.mark.parametrize("hp", [1, 6])
def test_tiny_planner_rollout(ff, hp):
    from kv_cache_attention_ff_gb300 import synth
    cfg_id, fields, _ = CONFIGS["tiny"]
    fields = dict(fields, planner_block=3, planner_history=hp, n_stages=1)
    dev = torch.device("cuda:0")
    T, h, d = 16, 2, 64
    bank = ff.Bank(**fields)
    obank = fo.OracleBank(oracle_cfg(fields))
    nb = fo.num_planner_blocks(13, 4, 3)
    for b in range(nb):
        frames = fo.planner_block_anchors(b, 3, 4, 13)
        q, k, v = (synth.frames_tensor(cfg_id, 0, 50, t, frames, T, h, d, "normal") for t in range(3))
        out = torch.empty((len(frames) * T, h, d), dtype=torch.bfloat16, device=dev)
        bank.planner_attn(0, b, from_bits(q, dev), from_bits(k, dev), from_bits(v, dev), out)
        ref, ctx = obank.planner_attn(0, b, q, k, v, planner_block=3, planner_history=hp)
        torch.cuda.synchronize()
        mae, rl2, ok = compare_out(out, ref)
        assert ok, (b, mae, rl2)
        # the block's cache-extraction forward publishes its clean anchor KV
        ka = synth.frames_tensor(cfg_id, 0, synth.ANCHOR_STREAM, synth.K, frames, T, h, d, "normal")
        va = synth.frames_tensor(cfg_id, 0, synth.ANCHOR_STREAM, synth.V, frames, T, h, d, "normal")
        bank.anchor_publish(0, frames[0], len(frames), from_bits(ka, dev), from_bits(va, dev))
        obank.anchor_publish(0, frames[0], len(frames), ka, va)
    assert bank.error_poll() == 0
    bank.close()


def test_planner_missing_history_anchor(ff):
    fields = dict(CONFIGS["tiny"][1], planner_block=3, planner_history=6, n_stages=1)
    dev = torch.device("cuda:0")
    bank = ff.Bank(**fields)
    z = torch.zeros((16, 2, 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(ff.FFError) as ei:
        bank.planner_attn(0, 1, z, z, z, torch.empty_like(z))
    assert ei.value.code == "FF_ERR_ANCHOR_MISSING"
    with pytest.raises(ff.FFError) as ei:
        bank.planner_attn(0, 2, z, z, z, torch.empty_like(z))
    assert ei.value.code == "FF_ERR_ARG"
    bank.close()
    nop = ff.Bank(**dict(fields, planner_history=0))
    z3 = torch.zeros((48, 2, 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(ff.FFError) as ei:
        nop.planner_attn(0, 0, z3, z3, z3, torch.empty_like(z3))
    assert ei.value.code == "FF_ERR_ARG"
    nop.close()


def test_wan13b_planner_w_ctx_block(ff):
    """261 latents at the 1.3B 480p shape: block 8 attends over blocks 2..7 (18 anchor
    frames) plus its own 3 = W_ctx = 21 frames = 32760 keys; sampled rows of all heads."""
    from kv_cache_attention_ff_gb300 import synth
    cfg_id = 6
    fields = dict(CONFIGS["wan13b_480p"][1], total_frames=261, anchor_capacity=27, n_stages=1, planner_block=3,
                  planner_history=6)
    T, h, d = 1560, 12, 128
    dev = torch.device("cuda:0")
    bank = ff.Bank(**fields)
    obank = fo.OracleBank(oracle_cfg(fields))
    anchors = list(range(0, 261, 10))
    ka = synth.device_frames(cfg_id, 0, synth.ANCHOR_STREAM, synth.K, anchors, T, h, d, "ar")
    va = synth.device_frames(cfg_id, 0, synth.ANCHOR_STREAM, synth.V, anchors, T, h, d, "normal")
    # clean KV of blocks 2..7 (anchors 60..230)
    sl = slice(6 * T, 24 * T)
    bank.anchor_publish(0, 60, 18, ka[sl].contiguous(), va[sl].contiguous())
    obank.anchor_publish(0, 60, 18, to_bits(ka[sl]), to_bits(va[sl]))
    own = [240, 250, 260]
    q, k, v = (synth.device_frames(cfg_id, 0, 51, t, own, T, h, d, "ar" if t < 2 else "normal") for t in range(3))
    out = torch.empty_like(q)
    bank.planner_attn(0, 8, q, k, v, out)
    c = obank.cfg
    Ks, Vs = [], []
    for a in range(60, 240, 10):
        slt = obank.anchor[0][fo.anchor_slot(a, 10, 27)]
        Ks.append(slt.k)
        Vs.append(slt.v)
    Ks.append(fo.rope_k_bits(to_bits(k), fo.token_positions(own, 30, 52), d, 1e4))
    Vs.append(to_bits(v))
    K = fo.bf16_bits_to_f64(np.concatenate(Ks))
    V = fo.bf16_bits_to_f64(np.concatenate(Vs))
    assert K.shape[0] == 21 * T
    Q = fo.rope_q_f64(to_bits(q), fo.token_positions(own, 30, 52), d, 1e4)
    rng = np.random.default_rng(9)
    rows = np.unique(np.concatenate([[0, 127, 128, 4679], rng.choice(4680, 96, replace=False)]))
    ref = fo.attention_rows_f64(Q, K, V, rows)
    torch.cuda.synchronize()
    mae, rl2, ok = compare_out(out[torch.from_numpy(rows).to(dev)], ref)
    assert ok, (mae, rl2)
    assert c.anchor_capacity == 27
    assert bank.error_poll() == 0
    bank.close()
