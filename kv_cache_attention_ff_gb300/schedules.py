"""Per-chunk attention-call schedules of FlashForward and of the two
cache-update-only baselines the pages compare against.

FlashForward summary (onedev.kr/papers/332), section "무엇인가" (what it is):
Self-Forcing finishes a chunk and passes its clean output through the model
once more to build the cache; HiAR conditions on less-noisy context but
re-encodes at every denoising stage; both pay forwards that do not advance
the output latent.  Section "어떻게 동작하나": FlashForward's renderer has no
cache-update-only forward -- every one of its S stage forwards also publishes
the chunk's KV.

A schedule lists, for one chunk and one layer, the attention calls it makes:
("denoise", k) for stage k and ("reencode", k) for a cache-update-only forward.
Only the call structure is modelled here; every call has the steady renderer
shape, and the timing uses the library's own ff_render_attn.
"""
from __future__ import annotations


def flashforward(stages: int) -> list[tuple[str, int]]:
    return [("denoise", k) for k in range(stages)]


def self_forcing(stages: int) -> list[tuple[str, int]]:
    # one clean re-encode after the last stage
    return flashforward(stages) + [("reencode", stages)]


def hiar(stages: int) -> list[tuple[str, int]]:
    # a re-encode accompanies every denoising stage
    out = []
    for k in range(stages):
        out += [("denoise", k), ("reencode", k)]
    return out


SCHEDULES = {"flashforward": flashforward, "self_forcing": self_forcing, "hiar": hiar}


def cache_update_only_calls(schedule: list[tuple[str, int]]) -> int:
    return sum(1 for kind, _ in schedule if kind == "reencode")
