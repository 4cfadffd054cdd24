"""Seeded synthetic inputs shaped like the FlashForward renderer workloads.

This module holds no arithmetic of the method: it only draws random tensors
and rounds them to bf16 bit patterns.  Both the oracle-side tests and the CUDA
path consume its output, so it must stay free of imports from either.

Recipe (the pages use Wan2.1 latents at 480p/720p; no dataset is used):
* every draw comes from ``numpy.random.Generator(PCG64(SeedSequence([cfg_id,
  layer, stream, tensor, frame])))``; stream 0..S-1 = renderer stage, stream
  ``ANCHOR_STREAM`` = planner/anchor tensors; tensor 0/1/2 = Q/K/V;
* Q and K ("ar" mode) follow an AR(1) process over absolute latent frames,
  z_f = rho z_{f-1} + sqrt(1 - rho^2) eps_f with rho = 0.9 and z_0 = eps_0,
  then every (token, head) d-vector is scaled to unit RMS (QK-norm-like);
* V, and every tensor in "normal" mode, is N(0, 1) per frame;
* values are rounded from fp32 to bf16 (round to nearest even).
"""
from __future__ import annotations

import numpy as np

ANCHOR_STREAM = 99
Q, K, V = 0, 1, 2
RHO = 0.9


def _rng(cfg_id: int, layer: int, stream: int, tensor: int, frame: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([cfg_id, layer, stream, tensor, frame])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even of finite fp32 values to bf16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def _eps(cfg_id, layer, stream, tensor, frame, shape):
    return _rng(cfg_id, layer, stream, tensor, frame).standard_normal(shape, dtype=np.float32)


def frames_tensor(cfg_id: int, layer: int, stream: int, tensor: int, frames: list[int],
                  tokens: int, heads: int, head_dim: int, mode: str) -> np.ndarray:
    """bf16 bit patterns [len(frames) * tokens, heads, head_dim] for the given
    absolute latent frames (frame-major).

    mode "normal": iid N(0,1) per frame.  mode "ar": the AR(1) unit-RMS
    process described in the module docstring (needs every frame up to
    max(frames), so it is generated sequentially).
    """
    shape = (tokens, heads, head_dim)
    out = np.empty((len(frames) * tokens, heads, head_dim), dtype=np.uint16)
    if mode == "normal":
        for r, f in enumerate(frames):
            out[r * tokens:(r + 1) * tokens] = f32_to_bf16_bits(_eps(cfg_id, layer, stream, tensor, f, shape))
        return out
    if mode != "ar":
        raise ValueError(mode)
    want = {f: r for r, f in enumerate(frames)}
    z = None
    c = np.float32(np.sqrt(1.0 - RHO * RHO))
    for f in range(max(frames) + 1):
        e = _eps(cfg_id, layer, stream, tensor, f, shape)
        z = e if z is None else np.float32(RHO) * z + c * e
        if f in want:
            rms = np.sqrt(np.mean(z * z, axis=-1, keepdims=True, dtype=np.float32))
            r = want[f]
            out[r * tokens:(r + 1) * tokens] = f32_to_bf16_bits(z / rms)
    return out


class ARStream:
    """Sequential AR(1) generator that yields consecutive frames without
    regenerating the prefix (for full rollouts)."""

    def __init__(self, cfg_id, layer, stream, tensor, tokens, heads, head_dim):
        self.key = (cfg_id, layer, stream, tensor)
        self.shape = (tokens, heads, head_dim)
        self.f = 0
        self.z = None

    def next(self) -> np.ndarray:
        e = _eps(*self.key, self.f, self.shape)
        c = np.float32(np.sqrt(1.0 - RHO * RHO))
        self.z = e if self.z is None else np.float32(RHO) * self.z + c * e
        self.f += 1
        rms = np.sqrt(np.mean(self.z * self.z, axis=-1, keepdims=True, dtype=np.float32))
        return f32_to_bf16_bits(self.z / rms)


# ---------------------------------------------------------------------------
# Device-side generation (same recipe, torch's seeded CUDA generator) for the
# large workloads.  Consumers that need host copies (the oracle) copy these
# tensors back; the values never depend on the library under test.
# ---------------------------------------------------------------------------

def _seed(cfg_id, layer, stream, tensor, frame) -> int:
    return int(np.random.SeedSequence([cfg_id, layer, stream, tensor, frame]).generate_state(1, np.uint64)[0] >> 1)


def _bf16_torch(x):
    import torch
    u = x.contiguous().view(torch.int32).to(torch.int64) & 0xFFFFFFFF
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.to(torch.int32).to(torch.int16).view(torch.bfloat16)


class DeviceARStream:
    """Consecutive frames of one (cfg, layer, stream, tensor) process on the GPU,
    as bf16 tensors [tokens, heads, head_dim]; mode "ar" or "normal"."""

    def __init__(self, cfg_id, layer, stream, tensor, tokens, heads, head_dim, mode, device="cuda"):
        self.key = (cfg_id, layer, stream, tensor)
        self.shape = (tokens, heads, head_dim)
        self.mode = mode
        self.device = device
        self.f = 0
        self.z = None

    def _eps(self, f):
        import torch
        g = torch.Generator(device=self.device)
        g.manual_seed(_seed(*self.key, f))
        return torch.randn(self.shape, generator=g, device=self.device, dtype=torch.float32)

    def next(self):
        import torch
        e = self._eps(self.f)
        self.f += 1
        if self.mode == "normal":
            return _bf16_torch(e)
        c = float(np.float32(np.sqrt(1.0 - RHO * RHO)))
        self.z = e if self.z is None else self.z * RHO + e * c
        rms = torch.sqrt(torch.mean(self.z * self.z, dim=-1, keepdim=True))
        return _bf16_torch(self.z / rms)

    def frames(self, n):
        import torch
        return torch.cat([self.next() for _ in range(n)], dim=0)


def device_frames(cfg_id, layer, stream, tensor, frames, tokens, heads, head_dim, mode, device="cuda"):
    """bf16 [len(frames) * tokens, heads, head_dim] on the device for the given
    absolute frames (AR mode regenerates the prefix on the device)."""
    import torch
    s = DeviceARStream(cfg_id, layer, stream, tensor, tokens, heads, head_dim, mode, device)
    want = {f: r for r, f in enumerate(frames)}
    out = [None] * len(frames)
    if mode == "normal":
        for f, r in want.items():
            s.f = f
            out[r] = s.next()
    else:
        for f in range(max(frames) + 1):
            x = s.next()
            if f in want:
                out[want[f]] = x
    return torch.cat(out, dim=0)
