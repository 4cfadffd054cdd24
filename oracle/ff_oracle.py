"""Plain, slow, fp64 CPU oracle for FlashForward renderer bank attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
module: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code with the
CUDA library (no headers, tables, helpers or generators); inputs are plain
numpy arrays of bf16 bit patterns (``uint16``) produced elsewhere.

What it computes (sources are the FlashForward pages; the page titles are
abbreviated as follows):

* [FF-onedev]  "FlashForward가 디노이징 중 KV 캐시를 재사용해 자기회귀 영상 생성을
  가속한다" (onedev.kr/papers/332).
* [FF-hotpaper] "In-Flight KV Cache with Clean Anchors for Faster
  Autoregressive Video Diffusion" (hotpaper.ai/paper/2609.32540).
* [FF-aifeeds] "In-Flight KV Cache 与 Clean Anchors" (ai-feeds.com/i/paper/2609.32540).
* [FAST-AR]    the gist.science summary of FAST-AR (gist.science/ko/paper/2602.01801),
  used only for one softmax identity in the tests, never as a method step.

Renderer forward, [FF-onedev] section "어떻게 동작하나" (how it works), Eq. (2):
    (v_hat, K, V) = F_R(x, c, tau_k; A_Gamma(i), B_k^(i))
    B_k^(i+1)    = Tail_H(B_k^(i) U (i, K, V))
i.e. chunk i at stage k attends over the clean anchors chosen by Gamma(i),
the last H chunks published at the same stage, and itself; then its own K/V
joins the stage bank, which keeps only the newest H chunks.  The anchor
schedule (stride Delta, planner blocks of 3, 81 latents -> 27 chunks of 3)
and the hyper-parameters B_P = B_R = 3, Delta = 10, S = 4, W_ctx = 21, H = 5
come from [FF-onedev] section "무엇과 다른가" (how it differs).

Readings where the pages are silent (each is also listed in the design notes):
* Gamma(i): nearest anchor at or before the chunk's first frame and nearest at
  or after its last frame; an anchor index past the last latent is dropped; if
  both coincide the anchor is used once.
* A final chunk with fewer than B_R frames when N mod B_R != 0.
* RoPE: the three-axis (t, y, x) rotary embedding of the backbone the pages
  name (Wan2.1), pairs of adjacent channels, head dim split
  d - 4*floor(d/6) | 2*floor(d/6) | 2*floor(d/6), omega_j = theta^(-2j/d_axis),
  theta = 10000.  The pages only name RoPE ([FF-onedev] section "전제와 한계").
* Published K is RoPE(K) with a fixed fp64 arithmetic contract and one
  round-to-nearest-even to bf16; V is stored as given; Q for attention stays
  unrounded fp64 here.
* Softmax scale 1/sqrt(d); no mask inside the key set.

Parity status: every function below is pinned by tests under
``tests/test_oracle_*.py`` against closed forms, library routines, worked
tables, exact rational arithmetic or brute force.  What no test can tie to the
pages is the RoPE *layout* choice itself (which axis gets which channels): the
pages name RoPE but never print a layout, so the layout is a reading
("parity unpinned" with respect to the pages), while the functions that
implement it are pinned (identity at the origin, textbook values, axis and
frequency mapping, pair norms, the relative-position identity, the rounded
exact rotation).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# ---------------------------------------------------------------------------
# bf16 <-> fp64, written from the IEEE-754 definition (independent of any GPU
# conversion code).
# ---------------------------------------------------------------------------

BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def round_f64_to_bf16_value(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    bf16 has 8 significant bits and fp32's exponent range.  A finite v with
    v = m * 2**e (0.5 <= |m| < 1) has bf16 spacing 2**(e-8) in the normal
    range and 2**-133 in the subnormal range (|v| < 2**-126).  Scaling by that
    spacing is exact in fp64, ``np.round`` rounds half to even, and the
    product is scaled back exactly.  Results beyond the largest finite bf16
    become +-inf.  This is a single rounding from fp64 (no fp32 step).
    """
    v = np.asarray(v, dtype=np.float64)
    out = v.copy()
    fin = np.isfinite(v)
    x = v[fin]
    _, e = np.frexp(x)
    q = np.maximum(e - 8, -133)
    r = np.round(np.ldexp(x, -q))
    y = np.ldexp(r, q)
    y = np.where(np.abs(y) > BF16_MAX, np.copysign(np.inf, x), y)
    out[fin] = y
    return out


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """RNE of float64 to bf16, returned as uint16 bit patterns."""
    r = round_f64_to_bf16_value(v)
    # r is exactly representable in fp32 (bf16 is a subset), so this cast is exact.
    return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ---------------------------------------------------------------------------
# Schedule: chunks, Gamma(i), history, slots.
# [FF-onedev] "무엇과 다른가": 81 latent positions rendered as 27 chunks of
# 3 latents; anchors at {0, 10, ..., 80}; renderer history H chunks.
# [FF-onedev] "어떻게 동작하나" Eq. (2): Tail_H keeps the last H chunks.
# ---------------------------------------------------------------------------


def num_chunks(total_frames: int, chunk_frames: int) -> int:
    return -(-total_frames // chunk_frames)


def chunk_span(i: int, chunk_frames: int, total_frames: int) -> tuple[int, int]:
    """First and last latent frame of renderer chunk i (a short final chunk when
    total_frames is not a multiple of chunk_frames)."""
    s = chunk_frames * i
    e = min(s + chunk_frames - 1, total_frames - 1)
    if s > e:
        raise ValueError("chunk index past the end of the video")
    return s, e


def gamma(i: int, chunk_frames: int, stride: int, total_frames: int) -> list[int]:
    """Gamma(i): the left/right clean anchors conditioning chunk i.

    Left = largest multiple of the stride <= first frame, right = smallest
    multiple >= last frame; right is dropped if it lies past the last latent,
    and a coincident pair is used once.  Order: [left, right].
    """
    s, e = chunk_span(i, chunk_frames, total_frames)
    left = stride * (s // stride)
    right = stride * (-(-e // stride))
    out = [left]
    if right != left and right <= total_frames - 1:
        out.append(right)
    return out


def history_chunks(i: int, history: int) -> list[int]:
    """Chunks of B_k^(i), oldest first: max(0, i-H) .. i-1."""
    return list(range(max(0, i - history), i))


def bank_slot(i: int, history: int) -> int:
    return i % history


def anchor_slot(a: int, stride: int, capacity: int) -> int:
    return (a // stride) % capacity


# Planner blocks ([FF-onedev] "무엇과 다른가": the planner produces the clean
# anchors B_P at a time, history H_P blocks, context budget W_ctx; "어떻게 쓰나":
# planner blocks attend causally to the clean KV of the previous blocks).


def num_anchors(total_frames: int, stride: int) -> int:
    return (total_frames - 1) // stride + 1


def num_planner_blocks(total_frames: int, stride: int, block: int) -> int:
    return -(-num_anchors(total_frames, stride) // block)


def planner_block_anchors(b: int, block: int, stride: int, total_frames: int) -> list[int]:
    """Anchor frames produced by planner block b."""
    n = num_anchors(total_frames, stride)
    if not 0 <= b * block < n:
        raise ValueError("planner block past the last anchor")
    return [a * stride for a in range(b * block, min((b + 1) * block, n))]


def planner_history_blocks(b: int, history: int) -> list[int]:
    """Blocks whose clean KV planner block b attends to, oldest first."""
    return list(range(max(0, b - history), b))


# ---------------------------------------------------------------------------
# Rotary position embedding (reading: the backbone's three-axis RoPE).
# ---------------------------------------------------------------------------


def rope_axis_dims(d: int) -> tuple[int, int, int]:
    seg = d // 6
    return d - 4 * seg, 2 * seg, 2 * seg


def rope_pair_axis(d: int) -> list[tuple[int, int, int]]:
    """For each channel pair p = (2p, 2p+1) of a head: (axis, j, d_axis) with
    axis 0 = time, 1 = row (y), 2 = column (x)."""
    dt, dy, dx = rope_axis_dims(d)
    out = []
    for axis, da in enumerate((dt, dy, dx)):
        for j in range(da // 2):
            out.append((axis, j, da))
    assert len(out) == d // 2
    return out


def rope_omega(j: int, d_axis: int, theta: float) -> float:
    return theta ** (-(2 * j) / d_axis)


def rope_cos_sin(positions: np.ndarray, d: int, theta: float) -> tuple[np.ndarray, np.ndarray]:
    """cos/sin of every channel pair for tokens at (t, y, x) positions.

    positions: int array [n, 3].  Angle = fl64(pos_axis * omega_j); cos and sin
    come from the C library through ``math``.  Returns two float64 arrays
    [n, d/2].
    """
    pairs = rope_pair_axis(d)
    n = positions.shape[0]
    c = np.empty((n, d // 2))
    s = np.empty((n, d // 2))
    for p, (axis, j, da) in enumerate(pairs):
        omega = rope_omega(j, da, theta)
        col = positions[:, axis]
        uniq, inv = np.unique(col, return_inverse=True)
        cu = np.array([math.cos(float(int(u)) * omega) for u in uniq])
        su = np.array([math.sin(float(int(u)) * omega) for u in uniq])
        c[:, p] = cu[inv]
        s[:, p] = su[inv]
    return c, s


def token_positions(frames: list[int], frame_h: int, frame_w: int) -> np.ndarray:
    """(t, y, x) of every token of the given latent frames, frame-major, each
    frame row-major over (y, x); t is the absolute latent index."""
    T = frame_h * frame_w
    pos = np.empty((len(frames) * T, 3), dtype=np.int64)
    n = np.arange(T)
    for r, f in enumerate(frames):
        pos[r * T:(r + 1) * T, 0] = f
        pos[r * T:(r + 1) * T, 1] = n // frame_w
        pos[r * T:(r + 1) * T, 2] = n % frame_w
    return pos


def rope_rotate_f64(x: np.ndarray, c: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Rotate adjacent channel pairs: (a, b) -> (a c - b s, a s + b c), each
    product and the sum/difference rounded once in fp64 (no fused multiply-add).

    x: float64 [n, h, d]; c, s: [n, d/2] (broadcast over heads).
    """
    a = x[..., 0::2]
    b = x[..., 1::2]
    cc = c[:, None, :]
    ss = s[:, None, :]
    ac = a * cc
    bs = b * ss
    as_ = a * ss
    bc = b * cc
    out = np.empty_like(x)
    out[..., 0::2] = ac - bs
    out[..., 1::2] = as_ + bc
    return out


def rope_k_bits(k_bits: np.ndarray, positions: np.ndarray, d: int, theta: float) -> np.ndarray:
    """Published K: RoPE in fp64 then one RNE to bf16 (bit patterns)."""
    c, s = rope_cos_sin(positions, d, theta)
    return f64_to_bf16_bits(rope_rotate_f64(bf16_bits_to_f64(k_bits), c, s))


def rope_q_f64(q_bits: np.ndarray, positions: np.ndarray, d: int, theta: float) -> np.ndarray:
    c, s = rope_cos_sin(positions, d, theta)
    return rope_rotate_f64(bf16_bits_to_f64(q_bits), c, s)


# ---------------------------------------------------------------------------
# Attention: the plain definition, one head at a time.
# ---------------------------------------------------------------------------


def attention_f64(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float | None = None) -> np.ndarray:
    """O = softmax(Q K^T * scale) V per head.  q [nq, h, d], k/v [nk, h, d]."""
    d = q.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.empty((q.shape[0], q.shape[1], v.shape[-1]))
    for hh in range(q.shape[1]):
        S = (q[:, hh, :] @ k[:, hh, :].T) * scale
        S = S - S.max(axis=1, keepdims=True)
        P = np.exp(S)
        P = P / P.sum(axis=1, keepdims=True)
        out[:, hh, :] = P @ v[:, hh, :]
    return out


def attention_rows_f64(q: np.ndarray, k: np.ndarray, v: np.ndarray, rows: np.ndarray,
                       heads: np.ndarray | None = None) -> np.ndarray:
    """The same definition evaluated only for selected query rows (and heads):
    returns [len(rows), len(heads), d]."""
    if heads is None:
        heads = np.arange(q.shape[1])
    return attention_f64(q[rows][:, heads], k[:, heads], v[:, heads])


def packed_block_causal(cfg: "BankConfig", q_bits, k_bits, v_bits, anchor_k_bits, anchor_v_bits) -> np.ndarray:
    """Packed block-causal renderer forward of one stage ([FF-onedev] "어떻게 쓰나":
    the renderer as one block-causal forward, targets attending to Gamma(i)
    anchors and the previous H same-noise chunks): by definition the outputs of
    rendering chunks 0, 1, ... in order at that stage with every anchor resident.
    Inputs cover all frames ([N*T, h, d]) and all anchors ([A*T, h, d])."""
    c = cfg
    T = c.tokens_per_frame
    bank = OracleBank(BankConfig(**{**c.__dict__, "n_layers": 1, "n_stages": 1,
                                    "anchor_capacity": num_anchors(c.total_frames, c.anchor_stride)}))
    bank.anchor_publish(0, 0, num_anchors(c.total_frames, c.anchor_stride), anchor_k_bits, anchor_v_bits)
    outs = []
    for i in range(num_chunks(c.total_frames, c.chunk_frames)):
        s, e = chunk_span(i, c.chunk_frames, c.total_frames)
        sl = slice(s * T, (e + 1) * T)
        outs.append(bank.render(0, 0, i, q_bits[sl], k_bits[sl], v_bits[sl]).out)
    return np.concatenate(outs)


def attention_bruteforce(q, k, v, scale=None):
    """Pure-Python triple loop of the same definition (tiny inputs only)."""
    nq, h, d = len(q), len(q[0]), len(q[0][0])
    nk = len(k)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = [[[0.0] * len(v[0][0]) for _ in range(h)] for _ in range(nq)]
    for i in range(nq):
        for hh in range(h):
            logits = []
            for j in range(nk):
                acc = 0.0
                for t in range(d):
                    acc += float(q[i][hh][t]) * float(k[j][hh][t])
                logits.append(acc * scale)
            m = max(logits)
            w = [math.exp(x - m) for x in logits]
            z = sum(w)
            for t in range(len(v[0][0])):
                acc = 0.0
                for j in range(nk):
                    acc += w[j] * float(v[j][hh][t])
                out[i][hh][t] = acc / z
    return out


# ---------------------------------------------------------------------------
# The bank state machine.
# ---------------------------------------------------------------------------


class OracleError(Exception):
    def __init__(self, code: str, msg: str = ""):
        super().__init__(f"{code}: {msg}")
        self.code = code


@dataclass
class BankConfig:
    n_layers: int
    total_frames: int
    heads: int
    head_dim: int
    frame_h: int
    frame_w: int
    n_stages: int = 4
    history: int = 5
    chunk_frames: int = 3
    anchor_stride: int = 10
    anchor_capacity: int = 9
    rope_theta: float = 10000.0

    @property
    def tokens_per_frame(self) -> int:
        return self.frame_h * self.frame_w


@dataclass
class _Slot:
    tag: int = -1
    frames: int = 0
    k: np.ndarray | None = None   # uint16 [frames*T, h, d]
    v: np.ndarray | None = None


@dataclass
class RenderResult:
    out: np.ndarray            # float64 [frames*T, h, d]
    k_rot_bits: np.ndarray     # uint16, as published
    anchors: list[int]
    history: list[int]
    slot: int
    key_frames: int
    context_frames: list[int] = field(default_factory=list)  # absolute latent index of each context frame


class OracleBank:
    """Per-layer stage banks B_k (H slots each) and the clean-anchor ring A."""

    def __init__(self, cfg: BankConfig):
        self.cfg = cfg
        self.stage = [[[_Slot() for _ in range(cfg.history)] for _ in range(cfg.n_stages)]
                      for _ in range(cfg.n_layers)]
        self.anchor = [[_Slot() for _ in range(cfg.anchor_capacity)] for _ in range(cfg.n_layers)]
        self.next_chunk = [[0] * cfg.n_stages for _ in range(cfg.n_layers)]

    # Anchor publish: clean anchor KV from the planner's cache-extraction
    # forward ([FF-onedev] "무엇과 다른가"): K rotated at t = anchor frame, V as is.
    def anchor_publish(self, layer: int, first_anchor: int, n: int, k_bits, v_bits) -> None:
        c = self.cfg
        T = c.tokens_per_frame
        if n < 1 or first_anchor % c.anchor_stride or first_anchor + (n - 1) * c.anchor_stride > c.total_frames - 1:
            raise OracleError("FF_ERR_ARG", "bad anchor range")
        for j in range(n):
            a = first_anchor + j * c.anchor_stride
            pos = token_positions([a], c.frame_h, c.frame_w)
            kb = k_bits[j * T:(j + 1) * T]
            sl = self.anchor[layer][anchor_slot(a, c.anchor_stride, c.anchor_capacity)]
            sl.tag, sl.frames = a, 1
            sl.k = rope_k_bits(kb, pos, c.head_dim, c.rope_theta)
            sl.v = np.array(v_bits[j * T:(j + 1) * T], copy=True)

    def render(self, layer: int, stage: int, chunk: int, q_bits, k_bits, v_bits) -> RenderResult:
        c = self.cfg
        T = c.tokens_per_frame
        if chunk != self.next_chunk[layer][stage]:
            raise OracleError("FF_ERR_ORDER", f"expected chunk {self.next_chunk[layer][stage]}")
        s, e = chunk_span(chunk, c.chunk_frames, c.total_frames)
        own_frames = list(range(s, e + 1))
        anchors = gamma(chunk, c.chunk_frames, c.anchor_stride, c.total_frames)
        ctx_k, ctx_v, ctx_frames = [], [], []
        for a in anchors:
            sl = self.anchor[layer][anchor_slot(a, c.anchor_stride, c.anchor_capacity)]
            if sl.tag != a:
                raise OracleError("FF_ERR_ANCHOR_MISSING", f"anchor {a}")
            ctx_k.append(sl.k)
            ctx_v.append(sl.v)
            ctx_frames.append(a)
        hist = history_chunks(chunk, c.history)
        for j in hist:
            sl = self.stage[layer][stage][bank_slot(j, c.history)]
            assert sl.tag == j, "Tail_H invariant broken"
            ctx_k.append(sl.k)
            ctx_v.append(sl.v)
            hs, he = chunk_span(j, c.chunk_frames, c.total_frames)
            ctx_frames.extend(range(hs, he + 1))
        pos = token_positions(own_frames, c.frame_h, c.frame_w)
        k_rot = rope_k_bits(k_bits, pos, c.head_dim, c.rope_theta)
        q_rot = rope_q_f64(q_bits, pos, c.head_dim, c.rope_theta)
        ctx_k.append(k_rot)
        ctx_v.append(np.asarray(v_bits))
        ctx_frames.extend(own_frames)
        K = bf16_bits_to_f64(np.concatenate(ctx_k, axis=0))
        V = bf16_bits_to_f64(np.concatenate(ctx_v, axis=0))
        out = attention_f64(q_rot, K, V)
        # Publish after the context has been read: B_k^(i+1) = Tail_H(B_k^(i) U (i, K, V)).
        sl = self.stage[layer][stage][bank_slot(chunk, c.history)]
        sl.tag, sl.frames = chunk, len(own_frames)
        sl.k = k_rot
        sl.v = np.array(v_bits, copy=True)
        self.next_chunk[layer][stage] += 1
        assert K.shape[0] == len(ctx_frames) * T
        return RenderResult(out, k_rot, anchors, hist, bank_slot(chunk, c.history),
                            len(ctx_frames), ctx_frames)

    def render_context(self, layer: int, stage: int, chunk: int, q_bits, k_bits, v_bits):
        """Like ``render`` but returns (q_rot f64, K f64, V f64) instead of the
        attention output, without changing state: lets tests evaluate the
        definition on sampled rows of very large calls."""
        c = self.cfg
        if chunk != self.next_chunk[layer][stage]:
            raise OracleError("FF_ERR_ORDER", "")
        s, e = chunk_span(chunk, c.chunk_frames, c.total_frames)
        own = list(range(s, e + 1))
        ks, vs = [], []
        for a in gamma(chunk, c.chunk_frames, c.anchor_stride, c.total_frames):
            sl = self.anchor[layer][anchor_slot(a, c.anchor_stride, c.anchor_capacity)]
            if sl.tag != a:
                raise OracleError("FF_ERR_ANCHOR_MISSING", f"anchor {a}")
            ks.append(sl.k)
            vs.append(sl.v)
        for j in history_chunks(chunk, c.history):
            sl = self.stage[layer][stage][bank_slot(j, c.history)]
            assert sl.tag == j, "Tail_H invariant broken"
            ks.append(sl.k)
            vs.append(sl.v)
        pos = token_positions(own, c.frame_h, c.frame_w)
        k_rot = rope_k_bits(k_bits, pos, c.head_dim, c.rope_theta)
        ks.append(k_rot)
        vs.append(np.asarray(v_bits))
        q = rope_q_f64(q_bits, pos, c.head_dim, c.rope_theta)
        return q, bf16_bits_to_f64(np.concatenate(ks)), bf16_bits_to_f64(np.concatenate(vs)), k_rot

    def commit_publish(self, layer: int, stage: int, chunk: int, k_rot_bits, v_bits) -> None:
        """State update of ``render`` alone (used with ``render_context``)."""
        c = self.cfg
        s, e = chunk_span(chunk, c.chunk_frames, c.total_frames)
        sl = self.stage[layer][stage][bank_slot(chunk, c.history)]
        sl.tag, sl.frames = chunk, e - s + 1
        sl.k = k_rot_bits
        sl.v = np.array(v_bits, copy=True)
        self.next_chunk[layer][stage] += 1

    def planner_attn(self, layer: int, block: int, q_bits, k_bits, v_bits, planner_block: int = 3,
                     planner_history: int = 6):
        """Attention of planner block `block`: its rotated queries over
        [clean anchor KV of the previous planner_history blocks; the block's own
        rotated K/V].  Publishes nothing.  Returns (out f64, context frames)."""
        c = self.cfg
        ks, vs, frames = [], [], []
        for hb in planner_history_blocks(block, planner_history):
            for a in planner_block_anchors(hb, planner_block, c.anchor_stride, c.total_frames):
                sl = self.anchor[layer][anchor_slot(a, c.anchor_stride, c.anchor_capacity)]
                if sl.tag != a:
                    raise OracleError("FF_ERR_ANCHOR_MISSING", f"anchor {a}")
                ks.append(sl.k)
                vs.append(sl.v)
                frames.append(a)
        own = planner_block_anchors(block, planner_block, c.anchor_stride, c.total_frames)
        pos = token_positions(own, c.frame_h, c.frame_w)
        ks.append(rope_k_bits(k_bits, pos, c.head_dim, c.rope_theta))
        vs.append(np.asarray(v_bits))
        frames.extend(own)
        q = rope_q_f64(q_bits, pos, c.head_dim, c.rope_theta)
        out = attention_f64(q, bf16_bits_to_f64(np.concatenate(ks)), bf16_bits_to_f64(np.concatenate(vs)))
        return out, frames

    def stage_tags(self, layer: int, stage: int) -> list[int]:
        return [sl.tag for sl in self.stage[layer][stage]]
