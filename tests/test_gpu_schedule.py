"""Parity of full schedules and long rollouts, concurrency across stage streams,
and the device-side failure-detection path."""
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


def _rows(nq, n, rng):
    fixed = [0, 127, 128, 255, 256, nq - 73, nq - 1]
    r = np.unique(np.concatenate([fixed, rng.choice(nq, n, replace=False)]))
    return r[r < nq]


def test_wan13b_480p_full_schedule_sampled(ff):
    """27 chunks x 4 stages x 30 layers, anchors first in 3 planner blocks; layers 0 and 29,
    stages 0 and 3 are checked: published K/V bytes at every chunk, attention on sampled
    rows at chunks 0-5, 13 and 26."""
    from kv_cache_attention_ff_gb300 import synth
    cfg_id, fields, mode = CONFIGS["wan13b_480p_schedule"]
    T, h, d = 1560, fields["heads"], fields["head_dim"]
    dev = torch.device("cuda:0")
    bank = ff.Bank(**fields)
    sampled, stages_chk, chunks_chk = (0, 29), (0, 3), {0, 1, 2, 3, 4, 5, 13, 26}
    obanks = {l: fo.OracleBank(oracle_cfg(dict(fields, n_layers=1))) for l in sampled}
    anchors = {}
    for l in sampled:
        anchors[l] = (synth.device_frames(cfg_id, l, synth.ANCHOR_STREAM, synth.K, list(range(0, 81, 10)), T, h, d,
                                          mode),
                      synth.device_frames(cfg_id, l, synth.ANCHOR_STREAM, synth.V, list(range(0, 81, 10)), T, h, d,
                                          "normal"))
    for layer in range(fields["n_layers"]):
        ka, va = anchors[layer if layer in anchors else 0]
        for b, (a0, n) in enumerate(anchor_blocks(fields)):
            sl = slice(3 * b * T, (3 * b + n) * T)
            bank.anchor_publish(layer, a0, n, ka[sl].contiguous(), va[sl].contiguous())
            if layer in obanks:
                obanks[layer].anchor_publish(0, a0, n, to_bits(ka[sl]), to_bits(va[sl]))
    streams = {(l, st): [synth.DeviceARStream(cfg_id, l, st, t, T, h, d, mode if t < 2 else "normal")
                         for t in (synth.Q, synth.K, synth.V)] for l in sampled for st in range(4)}
    rng = np.random.default_rng(3)
    out = torch.empty((3 * T, h, d), dtype=torch.bfloat16, device=dev)
    for i in range(27):
        s, e = fo.chunk_span(i, 3, 81)
        pos = fo.token_positions(list(range(s, e + 1)), 30, 52)
        for st in range(4):
            shared = [x.frames(3) for x in streams[(0, st)]]
            for layer in range(fields["n_layers"]):
                q, k, v = (shared if layer == 0 else
                           [x.frames(3) for x in streams[(layer, st)]] if layer in sampled else shared)
                bank.render_attn(layer, st, i, q, k, v, out)
                if layer not in sampled or st not in stages_chk:
                    continue
                ob = obanks[layer]
                qb, kb, vb = to_bits(q), to_bits(k), to_bits(v)
                if i in chunks_chk:
                    Q, K, V, k_rot = ob.render_context(0, st, i, qb, kb, vb)
                    rows = _rows(Q.shape[0], 48, rng)
                    ref = fo.attention_rows_f64(Q, K, V, rows)
                    torch.cuda.synchronize()
                    mae, rl2, ok = compare_out(out[torch.from_numpy(rows).to(dev)], ref)
                    assert ok, (layer, st, i, mae, rl2)
                else:
                    k_rot = fo.rope_k_bits(kb, pos, d, 10000.0)
                ob.commit_publish(0, st, i, k_rot, vb)
                torch.cuda.synchronize()
                tag, sk, sv = bank.slot_tensors(layer, st, i % 5)
                assert tag == i
                assert np.array_equal(to_bits(sk), k_rot) and np.array_equal(to_bits(sv), vb), (layer, st, i)
    assert bank.error_poll() == 0
    bank.close()


def _rollout_720p(ff, n_layers, layers):
    """261 latents = 87 chunks x 4 stages at 40 heads x 3600 tokens/frame, anchors
    published per planner block on demand into a 6-slot ring, rendered at the given
    layers of an n_layers-deep bank; bank bytes and device free memory stay constant
    over the rollout; stage 0 of every rendered layer checked: published K/V bytes at
    sampled chunks and attention on sampled rows of 4 heads at the last chunk."""
    from kv_cache_attention_ff_gb300 import synth
    cfg_id, fields, mode = CONFIGS["wan14b_720p_rollout"]
    fields = dict(fields, n_layers=n_layers)
    T, h, d = 3600, fields["heads"], fields["head_dim"]
    N = fields["total_frames"]
    dev = torch.device("cuda:0")
    bank = ff.Bank(**fields)
    bytes0 = bank.bytes()
    heads_chk = np.array([0, 13, 26, 39])
    # anchor stream: frames 0..260, keep the anchor frames
    ak = synth.DeviceARStream(cfg_id, 0, synth.ANCHOR_STREAM, synth.K, T, h, d, mode)
    av = synth.DeviceARStream(cfg_id, 0, synth.ANCHOR_STREAM, synth.V, T, h, d, "normal")
    anchor_k, anchor_v = {}, {}
    for f in range(N):
        kf = ak.next()
        if f % 10 == 0:
            anchor_k[f] = kf
        av.f = f
        if f % 10 == 0:
            anchor_v[f] = av.next()
    out = torch.empty((3 * T, h, d), dtype=torch.bfloat16, device=dev)
    chk_chunks = {0, 1, 2, 43, 86}
    rng = np.random.default_rng(5)
    for layer in layers:
        streams = [[synth.DeviceARStream(cfg_id, layer, st, t, T, h, d, mode if t < 2 else "normal")
                    for t in (synth.Q, synth.K, synth.V)] for st in range(4)]
        published = set()
        hist = {}       # stage-0 chunk -> (k bits, v bits) of the checked heads
        for i in range(87):
            for a in fo.gamma(i, 3, 10, N):
                blk = a // 30
                if blk not in published:
                    frames = [f for f in (30 * blk, 30 * blk + 10, 30 * blk + 20) if f < N]
                    kk = torch.cat([anchor_k[f] for f in frames])
                    vv = torch.cat([anchor_v[f] for f in frames])
                    bank.anchor_publish(layer, 30 * blk, len(frames), kk, vv)
                    published.add(blk)
            s, e = fo.chunk_span(i, 3, N)
            for st in range(4):
                q, k, v = (x.frames(3) for x in streams[st])
                torch.cuda.synchronize()
                free_a = torch.cuda.mem_get_info(dev)[0]
                bank.render_attn(layer, st, i, q, k, v, out)
                torch.cuda.synchronize()
                free_b = torch.cuda.mem_get_info(dev)[0]
                assert free_a == free_b, "the library allocated device memory during a render"
                assert bank.bytes() == bytes0
                if st != 0:
                    continue
                kb, vb = to_bits(k), to_bits(v)
                hist[i] = (kb[:, heads_chk], vb[:, heads_chk])
                hist.pop(i - 6, None)
                if i in chk_chunks:
                    pos = fo.token_positions(list(range(s, e + 1)), 45, 80)
                    k_rot = fo.rope_k_bits(kb, pos, d, 10000.0)
                    tag, sk, sv = bank.slot_tensors(layer, 0, i % 5)
                    assert tag == i and np.array_equal(to_bits(sk), k_rot) and np.array_equal(to_bits(sv), vb)
                if i == 86:
                    ks, vs = [], []
                    for a in fo.gamma(i, 3, 10, N):
                        pa = fo.token_positions([a], 45, 80)
                        ks.append(fo.rope_k_bits(to_bits(anchor_k[a])[:, heads_chk], pa, d, 10000.0))
                        vs.append(to_bits(anchor_v[a])[:, heads_chk])
                    for j in range(i - 5, i + 1):
                        js, je = fo.chunk_span(j, 3, N)
                        pj = fo.token_positions(list(range(js, je + 1)), 45, 80)
                        ks.append(fo.rope_k_bits(hist[j][0], pj, d, 10000.0))
                        vs.append(hist[j][1])
                    K = fo.bf16_bits_to_f64(np.concatenate(ks))
                    V = fo.bf16_bits_to_f64(np.concatenate(vs))
                    assert K.shape[0] == 72000
                    Q = fo.rope_q_f64(to_bits(q)[:, heads_chk], fo.token_positions(list(range(s, e + 1)), 45, 80), d,
                                      10000.0)
                    rows = _rows(Q.shape[0], 40, rng)
                    ref = fo.attention_rows_f64(Q, K, V, rows)
                    got = out[torch.from_numpy(rows).to(dev)][:, torch.from_numpy(heads_chk).to(dev)]
                    mae, rl2, ok = compare_out(got, ref)
                    assert ok, (layer, mae, rl2)
        assert len(published) == 9
    assert bank.error_poll() == 0
    nbytes = bank.bytes()
    bank.close()
    return nbytes


def test_wan14b_720p_rollout_constant_memory(ff):
    _rollout_720p(ff, 1, (0,))


def test_wan14b_720p_rollout_40_layer_bank(ff):
    """The 14B 720p bank at full depth: 40 layers x 4 stages of H + 1 = 6 ring slots of
    3 frames (K and V) plus 40 layers x 6 anchor slots; the rollout runs at layers 0
    and 39 with constant device memory at every call."""
    frame = 3600 * 40 * 128 * 2
    rings = 40 * 4 * 6 * 2 * 3 * frame
    anchors = 40 * 6 * 2 * frame
    assert (rings, anchors) == (212_336_640_000, 17_694_720_000)
    nbytes = _rollout_720p(ff, 40, (0, 39))
    scratch = nbytes - rings - anchors    # per-stage rotated-Q scratch and split partials, planner scratch, tables
    assert 0 < scratch < 2_000_000_000, scratch


def test_stage_streams_match_single_stream(ff):
    """Stages on their own CUDA streams (anchors on a fifth) give the same bytes as one stream."""
    from kv_cache_attention_ff_gb300 import synth
    cfg_id, fields, mode = CONFIGS["wan13b_480p"]
    fields = dict(fields, total_frames=36)
    T, h, d = 1560, 12, 128
    dev = torch.device("cuda:0")
    n_chunks = 12
    inputs = {(i, st): [synth.device_frames(cfg_id, 7, st, t, list(range(3 * i, 3 * i + 3)), T, h, d, "normal")
                        for t in range(3)] for i in range(n_chunks) for st in range(4)}
    ak = synth.device_frames(cfg_id, 7, synth.ANCHOR_STREAM, synth.K, [0, 10, 20, 30], T, h, d, "normal")
    av = synth.device_frames(cfg_id, 7, synth.ANCHOR_STREAM, synth.V, [0, 10, 20, 30], T, h, d, "normal")
    torch.cuda.synchronize()

    def run(streams):
        bank = ff.Bank(**dict(fields, anchor_capacity=4))
        outs = {}
        bank.anchor_publish(0, 0, 4, ak, av, streams[4])
        for i in range(n_chunks):
            for st in range(4):
                o = torch.empty((3 * T, h, d), dtype=torch.bfloat16, device=dev)
                q, k, v = inputs[(i, st)]
                bank.render_attn(0, st, i, q, k, v, o, streams[st])
                outs[(i, st)] = o
        torch.cuda.synchronize()
        slots = {(st, sl): bank.slot_tensors(0, st, sl)[1].clone() for st in range(4) for sl in range(5)}
        assert bank.error_poll() == 0
        bank.close()
        return outs, slots

    one = torch.cuda.Stream()
    a_out, a_slots = run([one] * 5)
    many = [torch.cuda.Stream() for _ in range(5)]
    b_out, b_slots = run(many)
    for key in a_out:
        assert torch.equal(a_out[key].view(torch.int16), b_out[key].view(torch.int16)), key
    for key in a_slots:
        assert torch.equal(a_slots[key], b_slots[key]), key


def test_device_wait_timeout_is_reported(ff):
    """A bounded device wait that runs out sets the error word; the host reads
    FF_ERR_DEVICE_TIMEOUT, the word clears, and the context keeps working."""
    fields = CONFIGS["tiny"][1]
    dev = torch.device("cuda:0")
    bank = ff.Bank(**fields)
    assert bank.error_poll() == 0
    bank.wait_probe(200)
    assert bank.error_poll() == 6
    assert bank.error_poll() == 0
    z = torch.zeros((3 * 16, 2, 64), dtype=torch.bfloat16, device=dev)
    bank.anchor_publish(0, 0, 2, torch.zeros((32, 2, 64), dtype=torch.bfloat16, device=dev),
                        torch.ones((32, 2, 64), dtype=torch.bfloat16, device=dev))
    out = torch.empty_like(z)
    bank.render_attn(0, 0, 0, z, z, torch.ones_like(z), out)
    torch.cuda.synchronize()
    assert torch.allclose(out.float(), torch.ones_like(out).float())
    assert bank.error_poll() == 0
    bank.close()
