"""ctypes binding of libff.so (argument marshalling only).

Every step of the renderer bank-attention path runs in the library's CUDA
kernels; this module only converts torch tensors and streams to pointers and
status codes to exceptions.  If the library is missing it raises: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libff.so")

FF_OK = 0
STATUS = {
    0: "FF_OK", 1: "FF_ERR_ARG", 2: "FF_ERR_ORDER", 3: "FF_ERR_ANCHOR_MISSING", 4: "FF_ERR_OOM",
    5: "FF_ERR_CUDA", 6: "FF_ERR_DEVICE_TIMEOUT", 7: "FF_ERR_UNSUPPORTED",
}

# Every entry point declared in include/ff.h.
EXPORTS = [
    "ff_desc_default", "ff_bank_create", "ff_anchor_publish", "ff_render_attn", "ff_bank_destroy",
    "ff_bank_gamma", "ff_bank_slot_info", "ff_bank_bytes", "ff_bank_error_poll", "ff_status_string",
    "ff_plan_chunk", "ff_bank_set_timing", "ff_bank_read_timing", "ff_render_kernel_count",
    "ff_attention_noalloc", "ff_bank_wait_probe", "ff_planner_attn", "ff_plan_planner_block",
    "ff_packed_workspace_bytes", "ff_packed_render_attn", "ff_render_attn_batch",
]


class FFError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        self.code = STATUS.get(status, str(status))
        super().__init__(f"{what}: {self.code} ({_lib().ff_status_string(status).decode()})")


class BankDesc(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int), ("n_stages", ctypes.c_int), ("history", ctypes.c_int),
        ("chunk_frames", ctypes.c_int), ("anchor_stride", ctypes.c_int), ("anchor_capacity", ctypes.c_int),
        ("total_frames", ctypes.c_int), ("heads", ctypes.c_int), ("head_dim", ctypes.c_int),
        ("frame_h", ctypes.c_int), ("frame_w", ctypes.c_int), ("rope_theta", ctypes.c_double),
        ("max_bytes", ctypes.c_size_t), ("device", ctypes.c_int), ("planner_block", ctypes.c_int),
        ("planner_history", ctypes.c_int),
    ]


class ChunkPlan(ctypes.Structure):
    _fields_ = [
        ("first_frame", ctypes.c_int), ("n_frames", ctypes.c_int), ("n_anchors", ctypes.c_int),
        ("anchors", ctypes.c_int * 2), ("n_hist", ctypes.c_int), ("hist_first", ctypes.c_int),
        ("hist_frames", ctypes.c_int), ("slot", ctypes.c_int), ("key_frames", ctypes.c_int),
    ]


class PlannerPlan(ctypes.Structure):
    _fields_ = [
        ("first_anchor", ctypes.c_int), ("n_anchors", ctypes.c_int), ("hist_first_block", ctypes.c_int),
        ("n_hist_blocks", ctypes.c_int), ("hist_frames", ctypes.c_int), ("key_frames", ctypes.c_int),
    ]


class KernelTimes(ctypes.Structure):
    _fields_ = [("calls", ctypes.c_int), ("publish_ms", ctypes.c_double), ("attn_ms", ctypes.c_double),
                ("combine_ms", ctypes.c_double), ("launches", ctypes.c_int)]


class RenderCall(ctypes.Structure):
    _fields_ = [("layer", ctypes.c_int), ("stage", ctypes.c_int), ("chunk", ctypes.c_int),
                ("q_pre", ctypes.c_void_p), ("k_pre", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("out", ctypes.c_void_p)]


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libff.so not built ({LIB_PATH}); run kv_cache_attention_ff_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, V = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
        lib.ff_desc_default.argtypes = [ctypes.POINTER(BankDesc)]
        lib.ff_bank_create.argtypes = [ctypes.POINTER(BankDesc), ctypes.POINTER(P)]
        lib.ff_anchor_publish.argtypes = [P, I, I, I, V, V, V]
        lib.ff_render_attn.argtypes = [P, I, I, I, V, V, V, V, V]
        lib.ff_bank_destroy.argtypes = [P]
        lib.ff_bank_gamma.argtypes = [P, I, ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(I)]
        lib.ff_bank_slot_info.argtypes = [P, I, I, I, ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(P),
                                          ctypes.POINTER(P)]
        lib.ff_bank_bytes.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
        lib.ff_bank_error_poll.argtypes = [P]
        lib.ff_status_string.argtypes = [I]
        lib.ff_status_string.restype = ctypes.c_char_p
        lib.ff_plan_chunk.argtypes = [ctypes.POINTER(BankDesc), I, ctypes.POINTER(ChunkPlan)]
        lib.ff_bank_set_timing.argtypes = [P, I]
        lib.ff_bank_read_timing.argtypes = [P, ctypes.POINTER(KernelTimes)]
        lib.ff_render_kernel_count.argtypes = [P, I, ctypes.POINTER(I)]
        lib.ff_attention_noalloc.argtypes = [V, V, V, V, I, I, I, I, V]
        lib.ff_bank_wait_probe.argtypes = [P, I, V]
        lib.ff_planner_attn.argtypes = [P, I, I, V, V, V, V, V]
        lib.ff_packed_workspace_bytes.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
        lib.ff_packed_render_attn.argtypes = [P, V, V, V, V, V, V, V, ctypes.c_size_t, V]
        lib.ff_plan_planner_block.argtypes = [ctypes.POINTER(BankDesc), I, ctypes.POINTER(PlannerPlan)]
        lib.ff_render_attn_batch.argtypes = [P, I, ctypes.POINTER(RenderCall), V]
        for name in EXPORTS:
            if name != "ff_status_string":
                getattr(lib, name).restype = ctypes.c_int
        _LIB = lib
    return _LIB


def lib():
    """The loaded ctypes library (raises ImportError if it was not built)."""
    return _lib()


def _check(status: int, what: str) -> None:
    if status != FF_OK:
        raise FFError(status, what)


def make_desc(**kw) -> BankDesc:
    d = BankDesc()
    _check(_lib().ff_desc_default(ctypes.byref(d)), "ff_desc_default")
    for k, v in kw.items():
        if not hasattr(d, k):
            raise TypeError(f"unknown bank field {k}")
        setattr(d, k, v)
    return d


def plan_chunk(desc: BankDesc, chunk: int) -> ChunkPlan:
    p = ChunkPlan()
    _check(_lib().ff_plan_chunk(ctypes.byref(desc), chunk, ctypes.byref(p)), "ff_plan_chunk")
    return p


def plan_planner_block(desc: BankDesc, block: int) -> PlannerPlan:
    p = PlannerPlan()
    _check(_lib().ff_plan_planner_block(ctypes.byref(desc), block, ctypes.byref(p)), "ff_plan_planner_block")
    return p


def attention_noalloc(q, k, v, out, stream=None):
    """Attention over a caller-held context without any device allocation
    (see ff_attention_noalloc in include/ff.h).  All four tensors must be on
    one device; the call runs with that device current."""
    import torch
    nq, heads, d = q.shape
    nk = k.shape[0]
    if any(t.device != q.device for t in (k, v, out)):
        raise ValueError("q, k, v and out must be on one device")
    if stream is not None and stream.device != q.device:
        raise ValueError("stream belongs to another device than the tensors")
    with torch.cuda.device(q.device):
        _check(_lib().ff_attention_noalloc(_ptr(q, (nq, heads, d), "q"), _ptr(k, (nk, heads, d), "k"),
                                           _ptr(v, (nk, heads, d), "v"), _ptr(out, (nq, heads, d), "out"),
                                           nq, nk, heads, d, _stream(stream, q.device)), "ff_attention_noalloc")


class _DevView:
    """__cuda_array_interface__ wrapper so torch can view bank memory without a copy."""

    def __init__(self, ptr: int, shape, device: int):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": "<u2", "data": (ptr, False),
                                         "version": 3, "strides": None}


def _ptr(t, shape, name):
    import torch
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous bf16 CUDA tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


class Bank:
    """Owner of one libff bank (stage banks, anchor ring and scratch of all layers)."""

    def __init__(self, **kw):
        self.desc = make_desc(**kw)
        self.handle = ctypes.c_void_p()
        _check(_lib().ff_bank_create(ctypes.byref(self.desc), ctypes.byref(self.handle)), "ff_bank_create")
        d = self.desc
        self.T = d.frame_h * d.frame_w
        self.device = d.device

    # -- core calls ---------------------------------------------------------
    def anchor_publish(self, layer, first_anchor_frame, n_anchors, k_pre, v, stream=None):
        shape = (n_anchors * self.T, self.desc.heads, self.desc.head_dim)
        _check(_lib().ff_anchor_publish(self.handle, layer, first_anchor_frame, n_anchors, _ptr(k_pre, shape, "k_pre"),
                                        _ptr(v, shape, "v"), _stream(stream, self.device)), "ff_anchor_publish")

    def render_attn(self, layer, stage, chunk, q_pre, k_pre, v, out, stream=None):
        frames = plan_chunk(self.desc, chunk).n_frames if 0 <= chunk < self.n_chunks else self.desc.chunk_frames
        shape = (frames * self.T, self.desc.heads, self.desc.head_dim)
        _check(_lib().ff_render_attn(self.handle, layer, stage, chunk, _ptr(q_pre, shape, "q_pre"),
                                     _ptr(k_pre, shape, "k_pre"), _ptr(v, shape, "v"), _ptr(out, shape, "out"),
                                     _stream(stream, self.device)), "ff_render_attn")

    def render_attn_batch(self, calls, stream=None):
        """Independent renderer calls, one per stage, issued together.
        `calls`: sequence of (layer, stage, chunk, q_pre, k_pre, v, out)."""
        arr = (RenderCall * len(calls))()
        for j, (layer, stage, chunk, q_pre, k_pre, v, out) in enumerate(calls):
            frames = plan_chunk(self.desc, chunk).n_frames if 0 <= chunk < self.n_chunks else self.desc.chunk_frames
            shape = (frames * self.T, self.desc.heads, self.desc.head_dim)
            arr[j] = RenderCall(layer, stage, chunk, _ptr(q_pre, shape, "q_pre"), _ptr(k_pre, shape, "k_pre"),
                                _ptr(v, shape, "v"), _ptr(out, shape, "out"))
        _check(_lib().ff_render_attn_batch(self.handle, len(calls), arr, _stream(stream, self.device)),
               "ff_render_attn_batch")

    def render_attn_batch_raw(self, calls, stream_handle) -> int:
        """Pointer-level batch: `calls` of (layer, stage, chunk, q_ptr, k_ptr, v_ptr, out_ptr); returns the status."""
        arr = (RenderCall * len(calls))(*[RenderCall(*c) for c in calls])
        return _lib().ff_render_attn_batch(self.handle, len(calls), arr, ctypes.c_void_p(stream_handle))

    def planner_attn(self, layer, block, q_pre, k_pre, v, out, stream=None):
        n = plan_planner_block(self.desc, block).n_anchors
        shape = (n * self.T, self.desc.heads, self.desc.head_dim)
        _check(_lib().ff_planner_attn(self.handle, layer, block, _ptr(q_pre, shape, "q_pre"), _ptr(k_pre, shape, "k_pre"),
                                      _ptr(v, shape, "v"), _ptr(out, shape, "out"), _stream(stream, self.device)),
               "ff_planner_attn")

    def packed_workspace_bytes(self) -> int:
        n = ctypes.c_size_t()
        _check(_lib().ff_packed_workspace_bytes(self.handle, ctypes.byref(n)), "ff_packed_workspace_bytes")
        return n.value

    def packed_render_attn(self, q_pre, k_pre, v, anchor_k_pre, anchor_v, out, workspace, stream=None):
        """All chunks of one stage in one block-causal call; `workspace` is a
        device uint8 tensor of at least packed_workspace_bytes()."""
        d = self.desc
        shape = (d.total_frames * self.T, d.heads, d.head_dim)
        ashape = (((d.total_frames - 1) // d.anchor_stride + 1) * self.T, d.heads, d.head_dim)
        if not workspace.is_cuda or workspace.numel() * workspace.element_size() < self.packed_workspace_bytes():
            raise ValueError("workspace too small")
        _check(_lib().ff_packed_render_attn(
            self.handle, _ptr(q_pre, shape, "q_pre"), _ptr(k_pre, shape, "k_pre"), _ptr(v, shape, "v"),
            _ptr(anchor_k_pre, ashape, "anchor_k_pre"), _ptr(anchor_v, ashape, "anchor_v"), _ptr(out, shape, "out"),
            ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size(),
            _stream(stream, self.device)), "ff_packed_render_attn")

    def render_attn_raw(self, layer, stage, chunk, q_ptr, k_ptr, v_ptr, out_ptr, stream_handle) -> int:
        """Pointer-level call (no checks in Python); returns the status code."""
        return _lib().ff_render_attn(self.handle, layer, stage, chunk, ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr),
                                     ctypes.c_void_p(v_ptr), ctypes.c_void_p(out_ptr), ctypes.c_void_p(stream_handle))

    def close(self):
        if self.handle:
            _lib().ff_bank_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- introspection ------------------------------------------------------
    @property
    def n_chunks(self):
        return -(-self.desc.total_frames // self.desc.chunk_frames)

    def gamma(self, chunk):
        l, r, n = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        _check(_lib().ff_bank_gamma(self.handle, chunk, ctypes.byref(l), ctypes.byref(r), ctypes.byref(n)),
               "ff_bank_gamma")
        return [l.value, r.value][:n.value]

    def slot_info(self, layer, stage, slot):
        tag, frames = ctypes.c_int(), ctypes.c_int()
        kp, vp = ctypes.c_void_p(), ctypes.c_void_p()
        _check(_lib().ff_bank_slot_info(self.handle, layer, stage, slot, ctypes.byref(tag), ctypes.byref(frames),
                                        ctypes.byref(kp), ctypes.byref(vp)), "ff_bank_slot_info")
        return tag.value, frames.value, kp.value, vp.value

    def slot_tensors(self, layer, stage, slot):
        """(tag, K, V) of a slot; K and V are uint16 (bf16 bit) views of bank memory."""
        import torch
        tag, frames, kp, vp = self.slot_info(layer, stage, slot)
        shape = (frames * self.T, self.desc.heads, self.desc.head_dim)
        if frames == 0:
            return tag, None, None
        with torch.cuda.device(self.device):
            k = torch.as_tensor(_DevView(kp, shape, self.device), device=f"cuda:{self.device}")
            v = torch.as_tensor(_DevView(vp, shape, self.device), device=f"cuda:{self.device}")
        return tag, k, v

    def bytes(self):
        n = ctypes.c_size_t()
        _check(_lib().ff_bank_bytes(self.handle, ctypes.byref(n)), "ff_bank_bytes")
        return n.value

    def error_poll(self):
        return _lib().ff_bank_error_poll(self.handle)

    def wait_probe(self, limit_ms: int, stream=None):
        """Enqueue the failure-detection self-test (a wait that times out)."""
        _check(_lib().ff_bank_wait_probe(self.handle, limit_ms, _stream(stream, self.device)), "ff_bank_wait_probe")

    def set_timing(self, enable: bool):
        _check(_lib().ff_bank_set_timing(self.handle, int(enable)), "ff_bank_set_timing")

    def read_timing(self) -> KernelTimes:
        t = KernelTimes()
        _check(_lib().ff_bank_read_timing(self.handle, ctypes.byref(t)), "ff_bank_read_timing")
        return t

    def kernel_count(self, chunk) -> int:
        c = ctypes.c_int()
        _check(_lib().ff_render_kernel_count(self.handle, chunk, ctypes.byref(c)), "ff_render_kernel_count")
        return c.value
