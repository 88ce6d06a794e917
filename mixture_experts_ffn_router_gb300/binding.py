"""ctypes binding of the C ABI in include/moe_ffn.h (argument marshalling only).

The functions keep the C names and take plain integers for device pointers and streams. ``MoeFFN``
is a small convenience wrapper that takes torch tensors (torch supplies device memory and the
stream; every step of the block runs in the library's kernels). Loading fails loudly when the
library has not been built: there is no fallback.
"""
import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe_ffn.so")

MOE_FFN_OK = 0
MOE_FFN_EINVAL = -1
MOE_FFN_EALIGN = -2
MOE_FFN_ETOOBIG = -3
MOE_FFN_EARCH = -4
MOE_FFN_ECUDA = -5
MOE_FFN_EDEVICE = -6
MOE_FFN_MOE_ONLY = 0
MOE_FFN_FULL_LAYER = 1
HIDDEN, N_EXPERTS, TOP_K, MOE_INTER, DENSE_INTER = 2816, 128, 8, 704, 2112
# Bits of the device status word (MOE_FFN_STATUS_* in include/moe_ffn.h).
STATUS_BITS = {"WAIT_FULL": 0x1, "WAIT_EMPTY": 0x2, "WAIT_ACC_FULL": 0x4, "WAIT_ACC_EMPTY": 0x8,
               "BAD_INDEX": 0x10, "BAD_SCHEDULE": 0x20, "DRAIN": 0x40, "WAIT_ITEM": 0x80,
               "WAIT_COPY": 0x100}


def decode_status(word: int) -> list:
    """Names of the bits set in a device status word, lowest first; unknown bits as hex."""
    names = [n for n, b in sorted(STATUS_BITS.items(), key=lambda kv: kv[1]) if word & b]
    rest = word & ~sum(STATUS_BITS.values())
    return names + (["0x%x" % rest] if rest else [])


KERNEL_NAMES = ("router_prep", "router_logits", "route_topk", "route_scatter", "gate_up_gemm", "down_gemm", "combine")
# Forwards of at most this many tokens run the whole routing front end (router sums, top-k,
# counting sort) as one kernel in slot 1; slots 0, 2 and 3 then launch nothing.
ROUTE_SMALL_T = 64


def slot_name(slot: int, T: int) -> str:
    """Name of the kernel a forward of T tokens launches in kernel slot `slot`."""
    if slot == 1 and T <= ROUTE_SMALL_T:
        return "route_small"
    return KERNEL_NAMES[slot]

_vp = ctypes.c_void_p


class moe_ffn_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("moe_inter", ctypes.c_int), ("dense_inter", ctypes.c_int), ("mode", ctypes.c_int),
                ("max_tokens", ctypes.c_int), ("eps", ctypes.c_float), ("router_scale", ctypes.c_float)]


WEIGHT_FIELDS = ("router_w", "router_norm_w", "per_expert_scale", "gate_up", "down", "dense_gate", "dense_up",
                 "dense_down", "pre_ff_ln", "pre_ff_ln_2", "post_ff_ln_1", "post_ff_ln_2", "post_ff_ln")


INT8_FIELDS = ("gate_up_q", "gate_up_scale", "down_q", "down_scale")
F4_FIELDS = ("gate_up_f4", "gate_up_f4s", "down_f4", "down_f4s")


class moe_ffn_weights(ctypes.Structure):
    _fields_ = ([(f, _vp) for f in WEIGHT_FIELDS] + [("layer_scalar", ctypes.c_float)] + [(f, _vp) for f in INT8_FIELDS]
                + [(f, _vp) for f in F4_FIELDS])


VIEW_FIELDS = ("logits", "topk_idx", "topk_w", "gap", "counts", "offsets", "perm", "w_sorted", "slot_pos", "n1",
               "n2", "h", "h_dense", "y", "d")


class moe_ffn_views(ctypes.Structure):
    _fields_ = [(f, _vp) for f in VIEW_FIELDS] + [("T", ctypes.c_int)]


_LIB = None


def lib():
    """The loaded CUDA library. Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmoe_ffn.so is not built (run __graft_entry__.build() or "
                               "python mixture_experts_ffn_router_gb300/build.py)")
        L = ctypes.CDLL(LIB_PATH)
        L.moe_ffn_workspace_bytes.restype = ctypes.c_size_t
        L.moe_ffn_workspace_bytes.argtypes = [ctypes.POINTER(moe_ffn_config)]
        L.moe_ffn_init.restype = ctypes.c_int
        L.moe_ffn_init.argtypes = [ctypes.POINTER(_vp), ctypes.POINTER(moe_ffn_config), _vp, ctypes.c_size_t,
                                   ctypes.c_int]
        L.moe_ffn_forward.restype = ctypes.c_int
        L.moe_ffn_forward.argtypes = [_vp, _vp, ctypes.c_int, ctypes.POINTER(moe_ffn_weights), _vp, _vp]
        L.moe_ffn_forward_shard.restype = ctypes.c_int
        L.moe_ffn_forward_shard.argtypes = [_vp, _vp, ctypes.c_int, ctypes.POINTER(moe_ffn_weights), ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, _vp, _vp, _vp]
        L.moe_ffn_finish_shards.restype = ctypes.c_int
        L.moe_ffn_finish_shards.argtypes = [_vp, _vp, ctypes.c_int, ctypes.POINTER(moe_ffn_weights), _vp, _vp, _vp,
                                            _vp]
        L.moe_ffn_workspace_view.restype = ctypes.c_int
        L.moe_ffn_workspace_view.argtypes = [_vp, ctypes.POINTER(moe_ffn_views)]
        L.moe_ffn_device_status.restype = ctypes.c_int
        L.moe_ffn_device_status.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_uint32)]
        L.moe_ffn_set_kernel_events.restype = ctypes.c_int
        L.moe_ffn_set_kernel_events.argtypes = [_vp, ctypes.c_int, _vp, _vp]
        L.moe_ffn_kernels_per_forward.restype = ctypes.c_int
        L.moe_ffn_kernels_per_forward.argtypes = [_vp, ctypes.c_int]
        L.moe_ffn_kernel_slots.restype = ctypes.c_int
        L.moe_ffn_kernel_slots.argtypes = [_vp, ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.c_int]
        L.moe_ffn_router_logits_noalloc.restype = ctypes.c_int
        L.moe_ffn_router_logits_noalloc.argtypes = [_vp, ctypes.c_int, _vp, _vp, ctypes.c_float, ctypes.c_float,
                                                     _vp, _vp]
        L.moe_ffn_selftest_wait_expiry.restype = ctypes.c_int
        L.moe_ffn_selftest_wait_expiry.argtypes = [_vp, _vp, _vp]
        L.moe_ffn_status_string.restype = ctypes.c_char_p
        L.moe_ffn_status_string.argtypes = [ctypes.c_int]
        L.moe_ffn_quantize_int8.restype = ctypes.c_int
        L.moe_ffn_quantize_int8.argtypes = [_vp, ctypes.c_longlong, ctypes.c_int, _vp, _vp, _vp]
        L.moe_ffn_quantize_mxfp4.restype = ctypes.c_int
        L.moe_ffn_quantize_mxfp4.argtypes = [_vp, ctypes.c_longlong, ctypes.c_int, _vp, _vp, _vp]
        L.moe_ffn_destroy.restype = None
        L.moe_ffn_destroy.argtypes = [_vp]
        _LIB = L
    return _LIB


class MoeFFNError(RuntimeError):
    def __init__(self, call, status):
        self.status = status
        super().__init__("%s: %s (%d)" % (call, moe_ffn_status_string(status), status))


def _check(call, status):
    if status != MOE_FFN_OK:
        raise MoeFFNError(call, status)
    return status


# ------------------------------------------------------------------ the C entry points

def moe_ffn_status_string(status: int) -> str:
    return lib().moe_ffn_status_string(int(status)).decode()


def make_config(mode: int, max_tokens: int, eps: float = 1e-6, router_scale: float = HIDDEN ** -0.5) -> moe_ffn_config:
    return moe_ffn_config(HIDDEN, N_EXPERTS, TOP_K, MOE_INTER, DENSE_INTER, int(mode), int(max_tokens),
                          float(eps), float(router_scale))


def moe_ffn_workspace_bytes(cfg: moe_ffn_config) -> int:
    return lib().moe_ffn_workspace_bytes(ctypes.byref(cfg))


def moe_ffn_init(cfg: moe_ffn_config, workspace: int, workspace_bytes: int, device: int) -> int:
    """Returns the context handle (an int)."""
    h = _vp()
    _check("moe_ffn_init", lib().moe_ffn_init(ctypes.byref(h), ctypes.byref(cfg), _vp(workspace),
                                               workspace_bytes, int(device)))
    return h.value


def moe_ffn_forward(ctx: int, x: int, T: int, weights: moe_ffn_weights, out: int, stream: int) -> int:
    return lib().moe_ffn_forward(_vp(ctx), _vp(x), int(T), ctypes.byref(weights), _vp(out), _vp(stream))


def moe_ffn_forward_shard(ctx: int, x: int, T: int, weights: moe_ffn_weights, expert_begin: int, expert_end: int,
                          with_dense: bool, moe_partial: int, dense_out: int, stream: int) -> int:
    return lib().moe_ffn_forward_shard(_vp(ctx), _vp(x), int(T), ctypes.byref(weights), int(expert_begin),
                                       int(expert_end), 1 if with_dense else 0, _vp(moe_partial), _vp(dense_out),
                                       _vp(stream))


def moe_ffn_finish_shards(ctx: int, x: int, T: int, weights: moe_ffn_weights, moe_sum: int, dense: int, out: int,
                          stream: int) -> int:
    return lib().moe_ffn_finish_shards(_vp(ctx), _vp(x), int(T), ctypes.byref(weights), _vp(moe_sum), _vp(dense),
                                       _vp(out), _vp(stream))


def expert_range(rank: int, world: int, n_experts: int = N_EXPERTS):
    """The contiguous experts [begin, end) that rank `rank` of `world` owns (equal shares, the first
    n_experts % world ranks one more)."""
    base, extra = divmod(n_experts, world)
    begin = rank * base + min(rank, extra)
    return begin, begin + base + (1 if rank < extra else 0)


def moe_ffn_workspace_view(ctx: int) -> moe_ffn_views:
    v = moe_ffn_views()
    _check("moe_ffn_workspace_view", lib().moe_ffn_workspace_view(_vp(ctx), ctypes.byref(v)))
    return v


def moe_ffn_device_status(ctx: int, stream: int):
    w = ctypes.c_uint32(0)
    rc = lib().moe_ffn_device_status(_vp(ctx), _vp(stream), ctypes.byref(w))
    return rc, w.value


def moe_ffn_set_kernel_events(ctx: int, kernel: int, start: int, stop: int) -> int:
    return lib().moe_ffn_set_kernel_events(_vp(ctx), int(kernel), _vp(start), _vp(stop))


def moe_ffn_kernels_per_forward(ctx: int, T: int) -> int:
    return lib().moe_ffn_kernels_per_forward(_vp(ctx), int(T))


def moe_ffn_kernel_slots(ctx: int, T: int) -> list:
    """The kernel slots a forward of T tokens launches, in launch order."""
    buf = (ctypes.c_int * len(KERNEL_NAMES))()
    n = lib().moe_ffn_kernel_slots(_vp(ctx), int(T), buf, len(KERNEL_NAMES))
    if n < 0:
        raise MoeFFNError("moe_ffn_kernel_slots", n)
    return list(buf[:n])


def moe_ffn_router_logits_noalloc(x: int, T: int, router_w: int, router_norm_w: int, router_scale: float,
                                  eps: float, logits: int, stream: int) -> int:
    """Router logits [T, 128] fp32 without any device allocation by the library (for callers that
    cannot allocate); its scratch is a fixed array shared by all calls, see include/moe_ffn.h."""
    return lib().moe_ffn_router_logits_noalloc(_vp(x), int(T), _vp(router_w), _vp(router_norm_w),
                                               float(router_scale), float(eps), _vp(logits), _vp(stream))


def moe_ffn_selftest_wait_expiry(status_word: int, record: int, stream: int) -> int:
    return lib().moe_ffn_selftest_wait_expiry(_vp(status_word), _vp(record), _vp(stream))


def moe_ffn_quantize_int8(w: int, rows: int, cols: int, q: int, scale: int, stream: int) -> int:
    return lib().moe_ffn_quantize_int8(_vp(w), int(rows), int(cols), _vp(q), _vp(scale), _vp(stream))


def quantize_experts_int8(w: dict) -> dict:
    """Adds the int8 form of the experts (gate_up_q/scale, down_q/scale) to a dict of CUDA weight
    tensors, made on the device by moe_ffn_quantize_int8."""
    import torch
    out = dict(w)
    s = torch.cuda.current_stream().cuda_stream
    for name, rows, cols in (("gate_up", N_EXPERTS * 2 * MOE_INTER, HIDDEN), ("down", N_EXPERTS * HIDDEN, MOE_INTER)):
        src = w[name]
        q = torch.empty((rows, cols), dtype=torch.int8, device=src.device)
        sc = torch.empty(rows, dtype=torch.float32, device=src.device)
        _check("moe_ffn_quantize_int8", moe_ffn_quantize_int8(src.data_ptr(), rows, cols, q.data_ptr(), sc.data_ptr(), s))
        out[name + "_q"] = q
        out[name + "_scale"] = sc
    return out


def moe_ffn_quantize_mxfp4(w: int, rows: int, cols: int, codes: int, scales: int, stream: int) -> int:
    return lib().moe_ffn_quantize_mxfp4(_vp(w), int(rows), int(cols), _vp(codes), _vp(scales), _vp(stream))


def quantize_experts_mxfp4(w: dict) -> dict:
    """Adds the MXFP4 form of the experts (gate_up_f4/f4s, down_f4/f4s) to a dict of CUDA weight
    tensors, made on the device by moe_ffn_quantize_mxfp4."""
    import torch
    out = dict(w)
    s = torch.cuda.current_stream().cuda_stream
    for name, rows, cols in (("gate_up", N_EXPERTS * 2 * MOE_INTER, HIDDEN), ("down", N_EXPERTS * HIDDEN, MOE_INTER)):
        src = w[name]
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=src.device)
        sc = torch.empty((rows, cols // 32), dtype=torch.uint8, device=src.device)
        _check("moe_ffn_quantize_mxfp4",
               moe_ffn_quantize_mxfp4(src.data_ptr(), rows, cols, codes.data_ptr(), sc.data_ptr(), s))
        out[name + "_f4"] = codes
        out[name + "_f4s"] = sc
    return out


def moe_ffn_destroy(ctx: int) -> None:
    lib().moe_ffn_destroy(_vp(ctx))


# ------------------------------------------------------------------ torch convenience layer

def _field_specs():
    """Element type and element count of every weight field, as include/moe_ffn.h states them."""
    import torch
    H, E, K2, I, D = HIDDEN, N_EXPERTS, 2 * MOE_INTER, MOE_INTER, DENSE_INTER
    f32, bf16, i8, u8 = torch.float32, torch.bfloat16, torch.int8, torch.uint8
    spec = {"router_w": (f32, E * H), "router_norm_w": (f32, H), "per_expert_scale": (f32, E),
            "gate_up": (bf16, E * K2 * H), "down": (bf16, E * H * I), "dense_gate": (bf16, D * H),
            "dense_up": (bf16, D * H), "dense_down": (bf16, H * D),
            "gate_up_q": (i8, E * K2 * H), "gate_up_scale": (f32, E * K2), "down_q": (i8, E * H * I),
            "down_scale": (f32, E * H), "gate_up_f4": (u8, E * K2 * H // 2), "gate_up_f4s": (u8, E * K2 * H // 32),
            "down_f4": (u8, E * H * I // 2), "down_f4s": (u8, E * H * I // 32)}
    for name in ("pre_ff_ln", "pre_ff_ln_2", "post_ff_ln_1", "post_ff_ln_2", "post_ff_ln"):
        spec[name] = (f32, H)
    return spec


def _check_type_size(what, t, dtype, numel):
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (what, dtype, t.dtype))
    if t.numel() != numel:
        raise ValueError("%s must hold %d elements, got %d" % (what, numel, t.numel()))


def _check_placement(what, t):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA tensor" % what)


def weights_struct(w: dict) -> moe_ffn_weights:
    """A moe_ffn_weights whose fields point at the CUDA tensors of ``w`` (absent fields are NULL).

    Each present tensor must have the field's element type and element count (include/moe_ffn.h),
    so that the kernels never read past a tensor that is too small. Types and sizes of all fields
    are checked before any placement, so a wrong one is named first."""
    spec = _field_specs()
    present = [(f, w[f]) for f in WEIGHT_FIELDS + INT8_FIELDS + F4_FIELDS if w.get(f) is not None]
    for f, t in present:
        _check_type_size("weight " + f, t, *spec[f])
    s = moe_ffn_weights()
    for f, t in present:
        _check_placement("weight " + f, t)
        setattr(s, f, t.data_ptr())
    if "layer_scalar" not in w:
        raise ValueError("layer_scalar is required")
    s.layer_scalar = float(w["layer_scalar"])
    return s


def check_io(x, out=None) -> int:
    """Checks a forward's input (and output, if given): contiguous bf16 CUDA tensors of shape
    [T, 2816], the output the same shape as the input. Returns T."""
    import torch
    if x.dim() != 2 or x.shape[1] != HIDDEN:
        raise ValueError("x must have shape [T, %d], got %s" % (HIDDEN, tuple(x.shape)))
    T = x.shape[0]
    _check_type_size("x", x, torch.bfloat16, T * HIDDEN)
    if out is not None:
        if tuple(out.shape) != tuple(x.shape):
            raise ValueError("out must have the shape of x %s, got %s" % (tuple(x.shape), tuple(out.shape)))
        _check_type_size("out", out, torch.bfloat16, T * HIDDEN)
    _check_placement("x", x)
    if out is not None:
        _check_placement("out", out)
    return T


class MoeFFN:
    """One context with its workspace (a torch uint8 tensor on the device)."""

    def __init__(self, mode: int, max_tokens: int, device: int = 0, workspace=None):
        import torch
        self.cfg = make_config(mode, max_tokens)
        self.nbytes = moe_ffn_workspace_bytes(self.cfg)
        if self.nbytes == 0:
            raise ValueError("invalid configuration")
        self.device = int(device)
        if workspace is None:
            workspace = torch.empty(self.nbytes, dtype=torch.uint8, device="cuda:%d" % self.device)
        elif workspace.numel() < self.nbytes:
            raise ValueError("workspace too small")
        self.workspace = workspace
        self.ctx = moe_ffn_init(self.cfg, workspace.data_ptr(), workspace.numel(), self.device)

    def forward(self, x, weights, out=None, stream=None):
        import torch
        T = check_io(x, out)
        if out is None:
            out = torch.empty_like(x)
        ws = weights if isinstance(weights, moe_ffn_weights) else weights_struct(weights)
        s = stream if stream is not None else torch.cuda.current_stream(x.device).cuda_stream
        _check("moe_ffn_forward", moe_ffn_forward(self.ctx, x.data_ptr(), T, ws, out.data_ptr(), s))
        return out

    def forward_shard(self, x, weights, expert_begin, expert_end, with_dense, stream=None):
        """One expert-parallel shard: (moe_partial, dense_out or None), fp32 [T, 2816] tensors."""
        import torch
        T = check_io(x)
        ws = weights if isinstance(weights, moe_ffn_weights) else weights_struct(weights)
        s = stream if stream is not None else torch.cuda.current_stream(x.device).cuda_stream
        part = torch.empty((T, HIDDEN), dtype=torch.float32, device=x.device)
        dense = torch.empty((T, HIDDEN), dtype=torch.float32, device=x.device) if with_dense else None
        _check("moe_ffn_forward_shard",
               moe_ffn_forward_shard(self.ctx, x.data_ptr(), T, ws, expert_begin, expert_end, with_dense,
                                     part.data_ptr(), dense.data_ptr() if dense is not None else 0, s))
        return part, dense

    def finish_shards(self, x, weights, moe_sum, dense, out=None, stream=None):
        """The block's output from the summed shard partials (and the shared-MLP output)."""
        import torch
        T = check_io(x, out)
        for name, t in (("moe_sum", moe_sum), ("dense", dense)):
            if t is not None:
                _check_type_size(name, t, torch.float32, T * HIDDEN)
                _check_placement(name, t)
        if out is None:
            out = torch.empty_like(x)
        ws = weights if isinstance(weights, moe_ffn_weights) else weights_struct(weights)
        s = stream if stream is not None else torch.cuda.current_stream(x.device).cuda_stream
        _check("moe_ffn_finish_shards",
               moe_ffn_finish_shards(self.ctx, x.data_ptr(), T, ws, moe_sum.data_ptr(),
                                     dense.data_ptr() if dense is not None else 0, out.data_ptr(), s))
        return out

    def views(self) -> moe_ffn_views:
        return moe_ffn_workspace_view(self.ctx)

    def status(self, stream=None):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        return moe_ffn_device_status(self.ctx, s)

    def close(self):
        if self.ctx:
            moe_ffn_destroy(self.ctx)
            self.ctx = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def view_tensor(ptr: int, shape, dtype, device: int = 0):
    """A torch tensor aliasing device memory at ``ptr`` (for reading the workspace views)."""
    import torch
    n = 1
    for s in shape:
        n *= s
    if n == 0:
        return torch.empty(shape, dtype=dtype, device="cuda:%d" % device)
    nbytes = n * torch.empty((), dtype=dtype).element_size()

    class _Holder:
        __cuda_array_interface__ = {
            "shape": (nbytes,), "typestr": "|u1", "data": (ptr, False), "version": 3, "strides": None,
        }

    raw = torch.as_tensor(_Holder(), device="cuda:%d" % device)
    return raw.view(dtype).view(*shape)
