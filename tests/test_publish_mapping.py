"""CPU check of the RoPE/publish kernel's thread -> unit mapping, restated from
kv_cache_attention_ff_gb300/csrc/ff_publish.cu: a thread handles the same 16-byte
unit of G consecutive heads of one token.  Every unit of a frame must be touched
exactly once, inside the frame, and the lanes of a warp must read whole head
rows for each of their G loads."""
import numpy as np
import pytest


def heads_per_thread(heads):
    return 2 if heads % 2 == 0 else 1


def thread_units(T, heads, head_dim):
    uph = head_dim // 8
    upr = heads * uph
    upf = T * upr
    G = heads_per_thread(heads)
    tid = np.arange(upf // G)
    o = tid & (uph - 1)
    rest = tid >> (uph.bit_length() - 1)
    groups = upr // (uph * G)
    tok = rest // groups
    off0 = tok * upr + (rest - tok * groups) * (G * uph) + o
    units = np.stack([off0 + j * uph for j in range(G)], axis=1)
    return units, upf, tok, o, uph, G


@pytest.mark.parametrize("T,heads,head_dim", [(16, 2, 64), (1560, 12, 128), (1560, 40, 128), (3600, 40, 128),
                                              (48, 1, 64), (40, 3, 128), (25, 3, 64)])
def test_every_unit_once_and_rows_coalesced(T, heads, head_dim):
    units, upf, tok, o, uph, G = thread_units(T, heads, head_dim)
    flat = units.ravel()
    assert flat.min() >= 0 and flat.max() < upf
    assert np.array_equal(np.sort(flat), np.arange(upf)), "a unit is missed or touched twice"
    # the G units of a thread are one token's heads at the same in-head offset (shared rotary angles)
    assert np.all(units // (heads * uph) == tok[:, None])
    assert np.all(units % uph == o[:, None])
    # per load j, lanes with the same (token, head group) read a contiguous head row
    for j in range(G):
        u = units[:, j]
        for w in range(0, min(len(u), 32 * 64), 32):
            lane = u[w:w + 32]
            runs = np.split(lane, np.where(np.diff(lane) != 1)[0] + 1)
            assert all(len(r) % min(uph, len(lane)) == 0 or len(r) == len(lane) for r in runs)
