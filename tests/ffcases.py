"""Workload definitions and helpers shared by the GPU parity tests, the smoke
check and the benchmark's baseline leg.

The configurations mirror the pages' workloads (FlashForward on Wan2.1,
onedev.kr/papers/332, "전제와 한계": 1.3B/14B backbones, 480p/720p, 81 latents
at 16 FPS and long rollouts); tensors are seeded synthetic stand-ins.
"""
from __future__ import annotations

import numpy as np

from oracle import ff_oracle as fo

# name -> (cfg_id, bank fields, input mode for Q/K)
CONFIGS = {
    "tiny": (1, dict(n_layers=1, n_stages=4, history=2, chunk_frames=3, anchor_stride=4, anchor_capacity=4,
                     total_frames=13, heads=2, head_dim=64, frame_h=4, frame_w=4), "normal"),
    "wan13b_480p": (2, dict(n_layers=1, n_stages=4, history=5, chunk_frames=3, anchor_stride=10, anchor_capacity=9,
                            total_frames=81, heads=12, head_dim=128, frame_h=30, frame_w=52), "ar"),
    "wan13b_480p_schedule": (3, dict(n_layers=30, n_stages=4, history=5, chunk_frames=3, anchor_stride=10,
                                     anchor_capacity=9, total_frames=81, heads=12, head_dim=128, frame_h=30,
                                     frame_w=52), "ar"),
    "wan14b_480p": (4, dict(n_layers=1, n_stages=4, history=5, chunk_frames=3, anchor_stride=10, anchor_capacity=9,
                            total_frames=81, heads=40, head_dim=128, frame_h=30, frame_w=52), "ar"),
    "wan14b_720p_rollout": (5, dict(n_layers=1, n_stages=4, history=5, chunk_frames=3, anchor_stride=10,
                                    anchor_capacity=6, total_frames=261, heads=40, head_dim=128, frame_h=45,
                                    frame_w=80), "ar"),
}


def oracle_cfg(fields: dict) -> fo.BankConfig:
    keys = ("n_layers", "total_frames", "heads", "head_dim", "frame_h", "frame_w", "n_stages", "history",
            "chunk_frames", "anchor_stride", "anchor_capacity")
    return fo.BankConfig(**{k: fields[k] for k in keys})


def to_bits(t) -> np.ndarray:
    """bf16 torch tensor (any device) -> numpy uint16 bit patterns."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits(a: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def compare_out(got_bf16, ref_f64: np.ndarray, max_abs=2e-2, rel_l2=5e-3):
    """Tolerances of the attention output against the fp64 definition."""
    import torch
    g = got_bf16.detach().to(torch.float64).cpu().numpy()
    diff = g - ref_f64
    mae = float(np.max(np.abs(diff)))
    rl2 = float(np.linalg.norm(diff) / max(np.linalg.norm(ref_f64), 1e-300))
    return mae, rl2, (mae <= max_abs and rl2 <= rel_l2)


def anchor_blocks(fields: dict):
    """Planner blocks of 3 anchors: (first frame, count), in order."""
    d, n = fields["anchor_stride"], fields["total_frames"]
    anchors = list(range(0, n, d))
    return [(anchors[j], len(anchors[j:j + 3])) for j in range(0, len(anchors), 3)]
