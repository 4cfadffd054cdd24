"""Call-structure model of FlashForward vs the cache-update-only baselines."""
from kv_cache_attention_ff_gb300 import schedules as sc


def test_call_counts_follow_the_pages():
    S = 4
    ff, sf, hi = sc.flashforward(S), sc.self_forcing(S), sc.hiar(S)
    # FlashForward: S forwards per chunk, none of them cache-update-only
    assert len(ff) == S and sc.cache_update_only_calls(ff) == 0
    # Self-Forcing: one clean re-encode per completed chunk
    assert sc.cache_update_only_calls(sf) == 1 and len(sf) == S + 1
    # HiAR: a re-encode at every denoising stage
    assert sc.cache_update_only_calls(hi) == S and len(hi) == 2 * S
    assert [k for kind, k in hi if kind == "denoise"] == list(range(S))
