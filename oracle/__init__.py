"""The oracle: a plain, slow CPU implementation of the Gemma-4 26B-A4B dual-path feed-forward block.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA path. The arithmetic lives
in ``moe_oracle.c`` (sources and precision are stated in ``moe_oracle.h``); this module only
marshals numpy arrays into it.

Pins (what the oracle is checked against, in ``tests/test_oracle_pins.py``):
  * GELU-tanh: its odd-part identity gelu(x) - gelu(-x) = x, its distance to the erf GELU (below
    4.73e-4 everywhere), torch's tanh-approximate gelu in fp64, and its special values.
  * RMSNorm: the constant-vector closed form and torch's rms_norm in fp64.
  * Router: softmax / top-k / renormalisation against a float64 full sort and torch.topk;
    renormalised weights sum to 1.
  * Expert MLP: identical experts reduce the expert branch to one plain MLP (torch, fp64).
  * The sparse == dense-masked identity of the 26B-A4B post ("The traceable trick"), bitwise.
  * The whole layer on tiny shapes against an independent float64 numpy brute force (brute.py).
  * The permutation against a brute-force sort of the slots by (expert, token).
  * int8 experts: the quantiser's error bound, symmetry, exact rows and zero rows; the layer with
    int8 experts against brute.py on the dequantised weights.
  * MXFP4 experts (``tests/test_oracle_fp4.py``): the shared-exponent rule (every block's maximum
    lands in [4, 8) scale units), exact grid values, the per-interval error bound and saturation,
    ties to the even code, symmetry, zero blocks; the layer with MXFP4 experts against brute.py on
    the dequantised weights.
  * The pins themselves: ``tests/test_oracle_mutants.py`` plants one plausible mistake at a time in
    a copy of ``moe_oracle.c`` and requires the pin files to fail on each.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None

_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u16p = ctypes.POINTER(ctypes.c_uint16)


class Dims(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int),
        ("n_experts", ctypes.c_int),
        ("top_k", ctypes.c_int),
        ("moe_inter", ctypes.c_int),
        ("dense_inter", ctypes.c_int),
        ("full_layer", ctypes.c_int),
        ("router_reads_pre2", ctypes.c_int),
        ("eps", ctypes.c_float),
        ("router_scale", ctypes.c_float),
    ]


class Weights(ctypes.Structure):
    _fields_ = [
        ("router_w", _f32p),
        ("router_norm_w", _f32p),
        ("per_expert_scale", _f32p),
        ("gate_up", _u16p),
        ("down", _u16p),
        ("dense_gate", _u16p),
        ("dense_up", _u16p),
        ("dense_down", _u16p),
        ("pre_ff_ln", _f32p),
        ("pre_ff_ln_2", _f32p),
        ("post_ff_ln_1", _f32p),
        ("post_ff_ln_2", _f32p),
        ("post_ff_ln", _f32p),
        ("layer_scalar", ctypes.c_float),
        ("gate_up_q", ctypes.POINTER(ctypes.c_int8)),
        ("gate_up_scale", _f32p),
        ("down_q", ctypes.POINTER(ctypes.c_int8)),
        ("down_scale", _f32p),
        ("gate_up_f4", ctypes.POINTER(ctypes.c_uint8)),
        ("gate_up_f4s", ctypes.POINTER(ctypes.c_uint8)),
        ("down_f4", ctypes.POINTER(ctypes.c_uint8)),
        ("down_f4s", ctypes.POINTER(ctypes.c_uint8)),
    ]


class Outputs(ctypes.Structure):
    _fields_ = [
        ("out", _f64p),
        ("moe", _f64p),
        ("dense", _f64p),
        ("h_slot", _f64p),
        ("y_slot", _f64p),
        ("h_dense", _f64p),
        ("logits", _f32p),
        ("probs", _f32p),
        ("topk_idx", _i32p),
        ("topk_w_renorm", _f32p),
        ("topk_w", _f32p),
        ("gap", _f32p),
    ]


def lib():
    """Loads (building first if needed) the oracle's shared library.

    MOE_ORACLE_LIB, when set, names another build of the same C source to load instead: the
    mutation test (tests/test_oracle_mutants.py) points it at copies with one planted mistake each
    and checks that the pins then fail.
    """
    global _LIB
    if _LIB is None:
        path = os.environ.get("MOE_ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        L.moe_oracle_gelu_tanh.restype = ctypes.c_double
        L.moe_oracle_gelu_tanh.argtypes = [ctypes.c_double]
        L.moe_oracle_rmsnorm.restype = None
        L.moe_oracle_rmsnorm.argtypes = [_f64p, _f32p, ctypes.c_int, ctypes.c_double, _f64p]
        L.moe_oracle_forward.restype = ctypes.c_int
        L.moe_oracle_forward.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, _u16p,
                                         ctypes.POINTER(Weights), ctypes.POINTER(Outputs), ctypes.c_int]
        L.moe_oracle_route.restype = ctypes.c_int
        L.moe_oracle_route.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, _u16p, ctypes.POINTER(Weights),
                                       ctypes.POINTER(Outputs)]
        L.moe_oracle_permute.restype = ctypes.c_int
        L.moe_oracle_permute.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, _f32p,
                                         _i32p, _i32p, _i32p, _f32p, _i32p]
        L.moe_oracle_quantize_int8.restype = ctypes.c_int
        L.moe_oracle_quantize_int8.argtypes = [_u16p, ctypes.c_longlong, ctypes.c_int,
                                               ctypes.POINTER(ctypes.c_int8), _f32p]
        L.moe_oracle_quantize_mxfp4.restype = ctypes.c_int
        L.moe_oracle_quantize_mxfp4.argtypes = [_u16p, ctypes.c_longlong, ctypes.c_int,
                                                ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(ctypes.c_uint8)]
        L.moe_oracle_set_threads.restype = None
        L.moe_oracle_set_threads.argtypes = [ctypes.c_int]
        L.moe_oracle_max_threads.restype = ctypes.c_int
        L.moe_oracle_max_threads.argtypes = []
        _LIB = L
    return _LIB


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _as(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError("expected %s, got %s" % (dtype, a.dtype))
    return a


def gelu_tanh(x: float) -> float:
    return lib().moe_oracle_gelu_tanh(float(x))


def rmsnorm(v, w, eps: float) -> np.ndarray:
    v = _as(np.asarray(v, dtype=np.float64), np.float64)
    w = _as(np.asarray(w, dtype=np.float32), np.float32)
    out = np.empty_like(v)
    lib().moe_oracle_rmsnorm(_ptr(v, ctypes.c_double), _ptr(w, ctypes.c_float), v.size, float(eps),
                             _ptr(out, ctypes.c_double))
    return out


def set_threads(n: int) -> None:
    lib().moe_oracle_set_threads(int(n))


def max_threads() -> int:
    return lib().moe_oracle_max_threads()


WEIGHT_FIELDS_F32 = ("router_w", "router_norm_w", "per_expert_scale", "pre_ff_ln", "pre_ff_ln_2",
                     "post_ff_ln_1", "post_ff_ln_2", "post_ff_ln")
WEIGHT_FIELDS_BF16 = ("gate_up", "down", "dense_gate", "dense_up", "dense_down")


def forward(dims: dict, x_bf16: np.ndarray, weights: dict, want=("out",), masked_dense=False,
            route_only=False) -> dict:
    """Runs the block on host arrays.

    dims: hidden, n_experts, top_k, moe_inter, dense_inter, full_layer, eps, router_scale and
      optionally router_reads_pre2. x_bf16: uint16 [T, H] (bf16 bit patterns). weights: numpy
      arrays, float32 for the fp32 fields and uint16 bf16 bit patterns for the bf16 fields (the
      dense and norm fields may be absent when full_layer is 0), plus the float layer_scalar.
    want: names of the outputs to return (fields of moe_oracle_outputs).
    route_only: run only the router (moe_oracle_route); only router outputs may be wanted.
    """
    H, E, K = dims["hidden"], dims["n_experts"], dims["top_k"]
    I, D = dims["moe_inter"], dims.get("dense_inter", 0)
    full = int(dims.get("full_layer", 0))
    x = _as(x_bf16, np.uint16).reshape(-1, H)
    T = x.shape[0]
    d = Dims(H, E, K, I, D if full else max(D, 1), full, int(dims.get("router_reads_pre2", 0)),
             float(dims["eps"]), float(dims["router_scale"]))
    keep = {}
    wst = Weights()
    for f in WEIGHT_FIELDS_F32:
        a = weights.get(f)
        if a is not None:
            a = _as(a, np.float32)
            keep[f] = a
            setattr(wst, f, _ptr(a, ctypes.c_float))
    for f in WEIGHT_FIELDS_BF16:
        a = weights.get(f)
        if a is not None:
            a = _as(a, np.uint16)
            keep[f] = a
            setattr(wst, f, _ptr(a, ctypes.c_uint16))
    for f in ("gate_up_q", "down_q"):
        a = weights.get(f)
        if a is not None:
            a = _as(a, np.int8)
            keep[f] = a
            setattr(wst, f, _ptr(a, ctypes.c_int8))
            sc = _as(weights[f.replace("_q", "_scale")], np.float32)
            keep[f.replace("_q", "_scale")] = sc
            setattr(wst, f.replace("_q", "_scale"), _ptr(sc, ctypes.c_float))
            keep.setdefault(f.replace("_q", ""), a)  # the bf16 form is not needed
    for f in ("gate_up_f4", "down_f4"):
        a = weights.get(f)
        if a is not None:
            a = _as(a, np.uint8)
            keep[f] = a
            setattr(wst, f, _ptr(a, ctypes.c_uint8))
            sc = _as(weights[f + "s"], np.uint8)
            keep[f + "s"] = sc
            setattr(wst, f + "s", _ptr(sc, ctypes.c_uint8))
            keep.setdefault(f.replace("_f4", ""), a)  # the bf16 form is not needed
    wst.layer_scalar = float(weights.get("layer_scalar", 1.0))
    if route_only:
        missing = [f for f in ("router_w", "router_norm_w", "per_expert_scale") if f not in keep]
        if full and dims.get("router_reads_pre2", 0) and "pre_ff_ln_2" not in keep:
            missing.append("pre_ff_ln_2")
    elif full:
        missing = [f for f in WEIGHT_FIELDS_F32 + WEIGHT_FIELDS_BF16 if f not in keep]
    else:
        missing = [f for f in ("router_w", "router_norm_w", "per_expert_scale", "gate_up", "down") if f not in keep]
    if missing:
        raise ValueError("missing weights: %s" % missing)

    shapes = {
        "out": ((T, H), np.float64), "moe": ((T, H), np.float64), "dense": ((T, H), np.float64),
        "h_slot": ((T, K, I), np.float64), "y_slot": ((T, K, H), np.float64),
        "h_dense": ((T, max(D, 1)), np.float64), "logits": ((T, E), np.float32),
        "probs": ((T, E), np.float32), "topk_idx": ((T, K), np.int32),
        "topk_w_renorm": ((T, K), np.float32), "topk_w": ((T, K), np.float32), "gap": ((T,), np.float32),
    }
    res = {}
    ost = Outputs()
    for name in want:
        shape, dt = shapes[name]
        a = np.zeros(shape, dtype=dt)
        res[name] = a
        ctype = {np.float64: ctypes.c_double, np.float32: ctypes.c_float, np.int32: ctypes.c_int32}[dt]
        setattr(ost, name, _ptr(a, ctype))
    if route_only:
        rc = lib().moe_oracle_route(ctypes.byref(d), T, _ptr(x, ctypes.c_uint16), ctypes.byref(wst),
                                    ctypes.byref(ost))
    else:
        rc = lib().moe_oracle_forward(ctypes.byref(d), T, _ptr(x, ctypes.c_uint16), ctypes.byref(wst),
                                      ctypes.byref(ost), 1 if masked_dense else 0)
    if rc != 0:
        raise RuntimeError("moe_oracle_forward failed (%d)" % rc)
    return res


def quantize_int8(w_bf16: np.ndarray):
    """Per-channel (per-row) symmetric int8 quantisation of a bf16 matrix (see
    moe_oracle_quantize_int8). Returns (q int8 [rows, cols], scale float32 [rows])."""
    w = _as(np.asarray(w_bf16), np.uint16)
    cols = w.shape[-1]
    rows = w.size // cols
    q = np.zeros(w.shape, np.int8)
    scale = np.zeros(rows, np.float32)
    rc = lib().moe_oracle_quantize_int8(_ptr(w, ctypes.c_uint16), rows, cols, _ptr(q, ctypes.c_int8),
                                        _ptr(scale, ctypes.c_float))
    if rc != 0:
        raise ValueError("moe_oracle_quantize_int8: bad arguments")
    return q, scale


def quantize_mxfp4(w_bf16: np.ndarray):
    """MXFP4 quantisation of a bf16 matrix [.., cols], cols a multiple of 32 (see
    moe_oracle_quantize_mxfp4). Returns (codes uint8 [rows, cols / 2], scales uint8 [rows, cols / 32])."""
    w = _as(np.asarray(w_bf16), np.uint16)
    cols = w.shape[-1]
    rows = w.size // cols
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows, max(cols // 32, 1)), np.uint8)
    rc = lib().moe_oracle_quantize_mxfp4(_ptr(w, ctypes.c_uint16), rows, cols, _ptr(codes, ctypes.c_uint8),
                                         _ptr(scales, ctypes.c_uint8))
    if rc != 0:
        raise ValueError("moe_oracle_quantize_mxfp4: bad arguments")
    return codes, scales


E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def dequantize_mxfp4(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """The float64 weights an MXFP4 matrix stands for (codes [rows, cols / 2], scales [rows, cols / 32])."""
    codes = np.asarray(codes, np.uint8)
    nib = np.stack([codes & 15, codes >> 4], axis=-1).reshape(codes.shape[0], -1)
    mag = E2M1[nib & 7]
    val = np.where(nib & 8, -mag, mag)
    e = np.repeat(np.asarray(scales, np.int64) - 127, 32, axis=1)
    return np.ldexp(val, e)


def permute(topk_idx: np.ndarray, topk_w, n_experts: int) -> dict:
    """Stable counting sort of the slots by expert (see moe_oracle_permute)."""
    idx = _as(np.asarray(topk_idx), np.int32)
    T, K = idx.shape
    S = T * K
    w = None if topk_w is None else _as(np.asarray(topk_w), np.float32)
    counts = np.zeros(n_experts, np.int32)
    offsets = np.zeros(n_experts + 1, np.int32)
    perm = np.zeros(S, np.int32)
    w_sorted = np.zeros(S, np.float32)
    slot_pos = np.zeros((T, K), np.int32)
    rc = lib().moe_oracle_permute(T, K, n_experts, _ptr(idx, ctypes.c_int32), _ptr(w, ctypes.c_float),
                                  _ptr(counts, ctypes.c_int32), _ptr(offsets, ctypes.c_int32),
                                  _ptr(perm, ctypes.c_int32), _ptr(w_sorted, ctypes.c_float),
                                  _ptr(slot_pos, ctypes.c_int32))
    if rc != 0:
        raise ValueError("moe_oracle_permute: expert id out of range")
    return {"counts": counts, "offsets": offsets, "perm": perm, "w_sorted": w_sorted, "slot_pos": slot_pos}


def gemma_dims(full_layer: bool) -> dict:
    """The 26B-A4B shapes ("Lab 008 — Raw lab detail", "The model under test")."""
    return {"hidden": 2816, "n_experts": 128, "top_k": 8, "moe_inter": 704, "dense_inter": 2112,
            "full_layer": int(bool(full_layer)), "eps": 1e-6, "router_scale": 2816 ** -0.5}


__all__ = ["lib", "gelu_tanh", "rmsnorm", "forward", "permute", "quantize_int8", "quantize_mxfp4",
           "dequantize_mxfp4", "set_threads", "max_threads",
           "gemma_dims", "Dims", "Weights", "Outputs"]
