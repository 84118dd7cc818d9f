"""Python binding of libmoe, the one-GPU MoE expert-parallel layer (include/moe.h).

Argument marshalling only: every step of dispatch -> grouped SwiGLU FFN -> combine runs in
the library's sm_103a kernels.  PyTorch provides device memory and the current stream.
There is no fallback: if libmoe.so is missing, or the device is not a GB300, the calls
raise.

Functions carry the C names: moe_workspace_size, moe_expert_out_size, moe_dispatch,
moe_prepare_weights, moe_expert_ffn, moe_combine, moe_get_status, and for the FP8 variant
moe_quantize_weights_fp8, moe_prepare_weights_fp8, moe_expert_ffn_fp8.  MoELayer1GPU
bundles them with the buffers of one geometry.
"""
import ctypes
import os

from .build import LIB_PATH, build  # noqa: F401

LAYOUT = {"EM": 0, "RM": 1, "FLAT": 2}
ALGO = {"LL": 0, "HT": 1}
QUANT = {"bf16": 0, "fp8": 1}
EXPERT_OUT = {"fp32": 0, "bf16": 1}
ACT = {"pair": 0, "bf16": 1}
IDS_INT32, IDS_INT64 = 0, 1
STATUS_BAD_EXPERT_ID, STATUS_EM_OVERFLOW, STATUS_TIMEOUT, STATUS_INACTIVE_RANK = 0x1, 0x2, 0x4, 0x8


class MoeGeom(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "world", "max_tok", "num_tokens", "hidden", "num_experts", "top_k", "intermediate",
        "layout", "algorithm", "quant", "expert_out_dtype", "act_precision")]


_P = ctypes.c_void_p
_HANDLE_PTRS = ("recv_x", "recv_scales", "counts", "offsets", "pick_pos", "pick_src", "slot",
                "layout_range", "recv_row", "recv_count", "num_recv", "recv_src", "recv_topk_idx",
                "recv_topk_weights", "status", "ffn_act", "ffn_act_scales", "pick_rows", "pick_row_scales",
                "workspace")


class MoeHandle(ctypes.Structure):
    _fields_ = ([("geom", MoeGeom)] + [(n, _P) for n in _HANDLE_PTRS] +
                [("workspace_bytes", ctypes.c_size_t), ("events", ctypes.POINTER(ctypes.c_void_p)),
                 ("num_events", ctypes.c_int32), ("magic", ctypes.c_uint64)])


# event slots of MoeHandle.events (MOE_EV_* in include/moe.h)
EV_DISPATCH_BEGIN, EV_ROUTING_END, EV_DISPATCH_END, EV_FFN_BEGIN, EV_GATHER_END, \
    EV_GEMM1_END, EV_GEMM2_END, EV_FFN_END, EV_COMBINE_BEGIN, EV_COMBINE_END = range(10)
EV_COUNT = 10


class MoeError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (where, strerror(code), code))


_lib = None


def lib():
    """The loaded libmoe.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmoe.so is not built (%s); run combine_topk_ids_gb300.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        G, H = ctypes.POINTER(MoeGeom), ctypes.POINTER(MoeHandle)
        sz = ctypes.POINTER(ctypes.c_size_t)
        L.moe_workspace_size.argtypes = [G, sz]
        L.moe_expert_out_size.argtypes = [G, sz]
        L.moe_dispatch.argtypes = [G, _P, _P, ctypes.c_int, _P, _P, _P, ctypes.c_size_t, H, _P]
        L.moe_prepare_weights.argtypes = [G, _P, _P, _P]
        L.moe_expert_ffn.argtypes = [H, _P, _P, _P, _P]
        L.moe_combine.argtypes = [H, _P, _P, _P, _P]
        L.moe_get_status.argtypes = [H, ctypes.POINTER(ctypes.c_int32), _P]
        L.moe_forward_host.argtypes = [G, _P, _P, ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                       _P, ctypes.c_size_t, H, _P]
        L.moe_launches_per_layer.argtypes = [G, ctypes.POINTER(ctypes.c_int32)]
        L.moe_launches_per_layer.restype = ctypes.c_int
        L.moe_route_noalloc.argtypes = [G, _P, ctypes.c_int] + [_P] * 8
        L.moe_route_noalloc.restype = ctypes.c_int
        L.moe_quantize_weights_fp8.argtypes = [G] + [_P] * 7
        L.moe_prepare_weights_fp8.argtypes = [G] + [_P] * 5
        L.moe_expert_ffn_fp8.argtypes = [H] + [_P] * 6
        L.moe_selftest_wait_expiry.argtypes = [_P, _P]
        L.moe_selftest_wait_expiry.restype = ctypes.c_int
        L.moe_strerror.argtypes = [ctypes.c_int]
        L.moe_strerror.restype = ctypes.c_char_p
        for f in ("moe_workspace_size", "moe_expert_out_size", "moe_dispatch",
                  "moe_prepare_weights", "moe_expert_ffn", "moe_combine", "moe_get_status",
                  "moe_forward_host", "moe_quantize_weights_fp8", "moe_prepare_weights_fp8",
                  "moe_expert_ffn_fp8"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().moe_strerror(int(code)).decode()


def _check(rc, where):
    if rc != 0:
        raise MoeError(rc, where)


def make_geom(W, Tr, T, H, E, k, I, layout="EM", algo="LL", quant="bf16", expert_out="fp32",
              act="pair") -> MoeGeom:
    return MoeGeom(W, Tr, T, H, E, k, I, LAYOUT[layout] if isinstance(layout, str) else layout,
                   ALGO[algo] if isinstance(algo, str) else algo,
                   QUANT[quant] if isinstance(quant, str) else quant,
                   EXPERT_OUT[expert_out] if isinstance(expert_out, str) else expert_out,
                   ACT[act] if isinstance(act, str) else act)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def moe_workspace_size(g: MoeGeom) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_workspace_size(ctypes.byref(g), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_expert_out_size(g: MoeGeom) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_expert_out_size(ctypes.byref(g), ctypes.byref(n)), "moe_expert_out_size")
    return n.value


def _ids_dtype(t):
    import torch
    return {torch.int64: IDS_INT64, torch.int32: IDS_INT32}.get(t.dtype, 99)


def moe_dispatch(g, x, topk_ids, topk_weights, workspace, stream=None, handle=None,
                 active_ranks=None) -> MoeHandle:
    """handle: optional MoeHandle to fill (its events fields are kept).  active_ranks: optional
    int32 [W] device tensor, 0 = failed logical rank."""
    h = MoeHandle() if handle is None else handle
    ids_dtype = _ids_dtype(topk_ids)
    _check(lib().moe_dispatch(ctypes.byref(g), _ptr(x), _ptr(topk_ids), ids_dtype,
                              _ptr(topk_weights), _ptr(active_ranks), _ptr(workspace),
                              workspace.numel() * workspace.element_size(),
                              ctypes.byref(h), _stream(stream)), "moe_dispatch")
    return h


def moe_prepare_weights(g, w1, w1_prepared, stream=None):
    _check(lib().moe_prepare_weights(ctypes.byref(g), _ptr(w1), _ptr(w1_prepared), _stream(stream)),
           "moe_prepare_weights")


def moe_expert_ffn(h, w1_prepared, w2, expert_out, stream=None):
    _check(lib().moe_expert_ffn(ctypes.byref(h), _ptr(w1_prepared), _ptr(w2), _ptr(expert_out),
                                _stream(stream)), "moe_expert_ffn")


def moe_quantize_weights_fp8(g, w1, w2, w1q_prepared, w1_scales_prepared, w2q, w2_scales, stream=None):
    _check(lib().moe_quantize_weights_fp8(ctypes.byref(g), _ptr(w1), _ptr(w2), _ptr(w1q_prepared),
                                          _ptr(w1_scales_prepared), _ptr(w2q), _ptr(w2_scales),
                                          _stream(stream)), "moe_quantize_weights_fp8")


def moe_prepare_weights_fp8(g, w1q, w1_scales, w1q_prepared, w1_scales_prepared, stream=None):
    _check(lib().moe_prepare_weights_fp8(ctypes.byref(g), _ptr(w1q), _ptr(w1_scales), _ptr(w1q_prepared),
                                         _ptr(w1_scales_prepared), _stream(stream)), "moe_prepare_weights_fp8")


def moe_expert_ffn_fp8(h, w1q_prepared, w1_scales_prepared, w2q, w2_scales, expert_out, stream=None):
    _check(lib().moe_expert_ffn_fp8(ctypes.byref(h), _ptr(w1q_prepared), _ptr(w1_scales_prepared), _ptr(w2q),
                                    _ptr(w2_scales), _ptr(expert_out), _stream(stream)), "moe_expert_ffn_fp8")


def moe_combine(h, expert_out, topk_weights, out, stream=None):
    _check(lib().moe_combine(ctypes.byref(h), _ptr(expert_out), _ptr(topk_weights), _ptr(out),
                             _stream(stream)), "moe_combine")


def moe_forward_host(g, x_host, ids_host, w_host, out_host, x_dev, ids_dev, w_dev, out_dev,
                     w1_prepared, w2, expert_out, workspace, handle, stream=None):
    """The whole layer from host buffers (torch CPU tensors), one C call.  With pinned
    (page-locked) host tensors the kernels read and write them directly and the device
    staging tensors may be None; otherwise they stage the copies."""
    import torch
    T, H, k = g.num_tokens, g.hidden, g.top_k
    cpu, cuda = torch.device("cpu"), torch.device("cuda")
    for t, name, dts, shape, dev in ((x_host, "x_host", (torch.bfloat16,), (T, H), cpu),
                                     (ids_host, "ids_host", (torch.int64, torch.int32), (T, k), cpu),
                                     (w_host, "w_host", (torch.float32,), (T, k), cpu),
                                     (out_host, "out_host", (torch.bfloat16,), (T, H), cpu),
                                     (x_dev, "x_dev", (torch.bfloat16,), (T, H), cuda),
                                     (ids_dev, "ids_dev", (getattr(ids_host, "dtype", torch.int64),), (T, k), cuda),
                                     (w_dev, "w_dev", (torch.float32,), (T, k), cuda),
                                     (out_dev, "out_dev", (torch.bfloat16,), (T, H), cuda)):
        if t is not None or dev is cpu:
            _require(t, name, dts, shape, dev)
    _check(lib().moe_forward_host(
        ctypes.byref(g), _ptr(x_host), _ptr(ids_host), _ids_dtype(ids_host), _ptr(w_host),
        _ptr(out_host), _ptr(x_dev), _ptr(ids_dev), _ptr(w_dev), _ptr(out_dev), _ptr(w1_prepared),
        _ptr(w2), _ptr(expert_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        ctypes.byref(handle), _stream(stream)), "moe_forward_host")


def moe_route_noalloc(g, topk_ids, counts, offsets, pick_pos, pick_src, slot, layout_range, status,
                      stream=None):
    """EXPERT_MAJOR routing into caller buffers with no workspace and no allocation, for
    callers that can only pass inputs and outputs (see include/moe.h)."""
    _check(lib().moe_route_noalloc(ctypes.byref(g), _ptr(topk_ids), _ids_dtype(topk_ids), _ptr(counts),
                                   _ptr(offsets), _ptr(pick_pos), _ptr(pick_src), _ptr(slot),
                                   _ptr(layout_range), _ptr(status), _stream(stream)),
           "moe_route_noalloc")


def moe_selftest_wait_expiry(status, stream=None):
    """Launch the bounded-wait expiry self-test (about 2 s on the device); status: int32
    device tensor that receives MOE_STATUS_TIMEOUT."""
    _check(lib().moe_selftest_wait_expiry(_ptr(status), _stream(stream)), "moe_selftest_wait_expiry")


def moe_launches_per_layer(g) -> int:
    n = ctypes.c_int32()
    _check(lib().moe_launches_per_layer(ctypes.byref(g), ctypes.byref(n)), "moe_launches_per_layer")
    return n.value


def moe_get_status(h, stream=None) -> int:
    v = ctypes.c_int32()
    _check(lib().moe_get_status(ctypes.byref(h), ctypes.byref(v), _stream(stream)), "moe_get_status")
    return v.value


def handle_view(h: MoeHandle, workspace, field: str, shape, dtype):
    """A torch view of one handle array (it lives inside `workspace`), for inspection."""
    import torch
    ptr = getattr(h, field)
    off = ptr - workspace.data_ptr()
    n = 1
    for s in shape:
        n *= s
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    return workspace.view(torch.uint8)[off:off + nbytes].view(dtype).view(*shape)


def _require(t, name, dtypes, shape, device):
    """Raise before any library call if `t` is not a contiguous tensor of one of `dtypes`
    and of `shape`, on `device` or in page-locked host memory (which the kernels read over
    the host link): the C ABI takes bare pointers and would read any other layout wrongly."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s: expected a torch.Tensor, got %s" % (name, type(t).__name__))
    if t.dtype not in dtypes:
        raise TypeError("%s: dtype %s, expected %s" % (name, t.dtype, " or ".join(str(d) for d in dtypes)))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s: shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    same = t.device.type == device.type and (device.index is None or t.device.index is None or
                                              t.device.index == device.index)
    if not same and not (t.device.type == "cpu" and t.is_pinned()):
        raise ValueError("%s is on %s; expected %s or page-locked host memory" % (name, t.device, device))


class MoELayer1GPU:
    """One MoE EP layer of a fixed geometry with its buffers on the current CUDA device.

    forward(x, topk_ids, topk_weights) = moe_dispatch -> moe_expert_ffn -> moe_combine,
    all on the current stream, no host synchronisation.  quant="fp8": FP8 dispatch and
    moe_expert_ffn_fp8 on weights quantised by set_weights.  expert_out="bf16": the expert
    stage's output (and the RANK_MAJOR / FLAT per-pick rows) in bf16.  act: the SwiGLU
    activation as the second GEMM's operand, "pair" (default: a bf16 (hi, lo) pair) or
    "bf16" (one bf16 value: faster, less accurate; see moe_act_precision in moe.h).
    """

    def __init__(self, W, Tr, T, H, E, k, I, layout="EM", algo="LL", device="cuda", quant="bf16",
                 expert_out="fp32", act="pair"):
        import torch
        self.quant = quant
        self.geom = make_geom(W, Tr, T, H, E, k, I, layout, algo, quant, expert_out, act)
        self.device = torch.device(device)
        self.workspace = torch.empty(moe_workspace_size(self.geom), dtype=torch.uint8, device=self.device)
        eo_t = torch.bfloat16 if expert_out == "bf16" else torch.float32
        self.expert_out = torch.empty(moe_expert_out_size(self.geom) // (2 if expert_out == "bf16" else 4),
                                      dtype=eo_t, device=self.device)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=self.device)
        self.w1p = None
        self.w2 = None
        self.handle = MoeHandle()
        self.events = None
        self._ev_array = None

    def enable_timing(self, on=True):
        """Record MOE_EV_* CUDA events between the kernels of every call (per-kernel times)."""
        import torch
        if not on:
            self.events, self._ev_array = None, None
            self.handle.events, self.handle.num_events = None, 0
            return
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(EV_COUNT)]
        for e in self.events:
            e.record()   # creates the underlying cudaEvent_t
        self._ev_array = (ctypes.c_void_p * EV_COUNT)(*[e.cuda_event for e in self.events])
        self.handle.events = ctypes.cast(self._ev_array, ctypes.POINTER(ctypes.c_void_p))
        self.handle.num_events = EV_COUNT

    def kernel_times_ms(self):
        """Per-kernel milliseconds of the last forward (enable_timing must be on)."""
        e = self.events
        t = lambda a, b: e[a].elapsed_time(e[b])  # noqa: E731
        em = self.geom.layout == LAYOUT["EM"]
        d = {"routing": t(EV_DISPATCH_BEGIN, EV_ROUTING_END),
             "dispatch_copy": t(EV_ROUTING_END, EV_DISPATCH_END),
             "gemm1_swiglu": t(EV_GATHER_END, EV_GEMM1_END),
             "gemm2": t(EV_GEMM1_END, EV_GEMM2_END),
             "combine": t(EV_COMBINE_BEGIN, EV_COMBINE_END)}
        if not em:
            d["reduce_ranks"] = t(EV_GEMM2_END, EV_FFN_END)
        d["dispatch"] = t(EV_DISPATCH_BEGIN, EV_DISPATCH_END)
        d["ffn"] = t(EV_FFN_BEGIN, EV_FFN_END)
        return d

    def set_weights(self, w1, w2):
        """bf16 w1 [E, 2I, H] and w2 [E, H, I]; prepared (FP8: quantised) once here."""
        import torch
        g = self.geom
        E, H, I = g.num_experts, g.hidden, g.intermediate
        _require(w1, "w1", (torch.bfloat16,), (E, 2 * I, H), self.device)
        _require(w2, "w2", (torch.bfloat16,), (E, H, I), self.device)
        if self.quant == "fp8":
            E, I2, H = w1.shape
            dev = w1.device
            self.w1p = torch.empty((E, I2, H), dtype=torch.uint8, device=dev)
            self.w1s = torch.empty((E, I2 // 128, H // 128), dtype=torch.float32, device=dev)
            self.w2 = torch.empty(tuple(w2.shape), dtype=torch.uint8, device=dev)
            self.w2s = torch.empty((E, H // 128, I2 // 256), dtype=torch.float32, device=dev)
            moe_quantize_weights_fp8(self.geom, w1, w2, self.w1p, self.w1s, self.w2, self.w2s)
            return
        self.w1p = torch.empty_like(w1)
        moe_prepare_weights(self.geom, w1, self.w1p)
        self.w2 = w2

    def _check_routing(self, topk_ids, topk_weights):
        import torch
        T, k = self.geom.num_tokens, self.geom.top_k
        _require(topk_ids, "topk_ids", (torch.int64, torch.int32), (T, k), self.device)
        _require(topk_weights, "topk_weights", (torch.float32,), (T, k), self.device)

    def dispatch(self, x, topk_ids, topk_weights, active_ranks=None):
        import torch
        _require(x, "x", (torch.bfloat16,), (self.geom.num_tokens, self.geom.hidden), self.device)
        self._check_routing(topk_ids, topk_weights)
        if active_ranks is not None:
            _require(active_ranks, "active_ranks", (torch.int32,), (self.geom.world,), self.device)
        moe_dispatch(self.geom, x, topk_ids, topk_weights, self.workspace, handle=self.handle,
                     active_ranks=active_ranks)
        return self.handle

    def expert_ffn(self):
        if self.w1p is None:
            raise RuntimeError("set_weights() has not been called")
        if self.quant == "fp8":
            moe_expert_ffn_fp8(self.handle, self.w1p, self.w1s, self.w2, self.w2s, self.expert_out)
        else:
            moe_expert_ffn(self.handle, self.w1p, self.w2, self.expert_out)
        return self.expert_out

    def combine(self, topk_weights):
        import torch
        _require(topk_weights, "topk_weights", (torch.float32,),
                 (self.geom.num_tokens, self.geom.top_k), self.device)
        moe_combine(self.handle, self.expert_out, topk_weights, self.out)
        return self.out

    def forward(self, x, topk_ids, topk_weights, active_ranks=None):
        self.dispatch(x, topk_ids, topk_weights, active_ranks)
        self.expert_ffn()
        return self.combine(topk_weights)

    def status(self) -> int:
        return moe_get_status(self.handle)

    def view(self, field, shape, dtype):
        return handle_view(self.handle, self.workspace, field, shape, dtype)
