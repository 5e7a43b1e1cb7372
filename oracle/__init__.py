"""CPU oracle for the SiTU routed-MoE expert layer (test infrastructure).

Only the tests, the package smoke check and the bench's CPU-baseline /
reference leg may import this package.  The product path (the CUDA library
and its binding) never does.  This module compiles ``situ_oracle.c`` with
gcc and exposes it through ctypes on numpy arrays; it shares no code with
the CUDA path.

The functions follow the pages they cite (see ``situ_oracle.c``):
  * ``quant_mxfp8``  -- per-token MXFP8 activation quantisation
    (TokenSpeed SiTU, "Supported contract" / "Activation precision").
  * ``permute``      -- expert permute with local-shard filtering
    (TokenSpeed SiTU, "Supported contract").
  * ``moe_forward``  -- the golden routed-MoE loop with SiTU
    (TensorRT-LLM PR #17865, golden ``_situ_act``) and the per-expert
    beta / up-half rescale (FlashInfer 0.6.18 MoE-LoRA AOT release notes,
    "Changes since 875b7d7").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "situ_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libsitu_oracle.so")
_lib = None
_lock = threading.Lock()

ACT_BF16, ACT_MXFP8, ACT_NVFP4 = 0, 1, 2
ACT_FN_SITU, ACT_FN_SWIGLU_BIAS = 0, 1
W_MXFP4, W_NVFP4 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (idempotent)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Args(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("T", "H", "I", "E_total", "E_loc", "off", "K", "act", "wt")] + [
        ("x_bf16", ctypes.c_void_p), ("x_q", ctypes.c_void_p), ("x_s", ctypes.c_void_p),
        ("x_gs", ctypes.c_void_p), ("ids", ctypes.c_void_p), ("wts", ctypes.c_void_p),
        ("w1", ctypes.c_void_p), ("w1s", ctypes.c_void_p), ("w1_gs", ctypes.c_void_p),
        ("w2", ctypes.c_void_p), ("w2s", ctypes.c_void_p), ("w2_gs", ctypes.c_void_p),
        ("beta", ctypes.c_void_p), ("beta_lin", ctypes.c_void_p),
        ("alpha_g", ctypes.c_void_p), ("alpha_u", ctypes.c_void_p), ("alpha2", ctypes.c_void_p),
        ("activation", ctypes.c_int), ("topk_in_fc1", ctypes.c_int), ("h1_nvfp4", ctypes.c_int),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            l = ctypes.CDLL(build())
            for name in ("oracle_e2m1_value", "oracle_e4m3_value", "oracle_ue8m0_value"):
                getattr(l, name).restype = ctypes.c_double
                getattr(l, name).argtypes = [ctypes.c_uint]
            l.oracle_bf16_value.restype = ctypes.c_double
            l.oracle_bf16_value.argtypes = [ctypes.c_uint16]
            l.oracle_f32_to_bf16.restype = ctypes.c_uint16
            l.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
            l.oracle_e4m3_encode.restype = ctypes.c_uint
            l.oracle_e4m3_encode.argtypes = [ctypes.c_double]
            l.oracle_mxfp8_exponent.restype = ctypes.c_int
            l.oracle_mxfp8_exponent.argtypes = [ctypes.c_double]
            l.oracle_situ.restype = ctypes.c_double
            l.oracle_situ.argtypes = [ctypes.c_double] * 4
            l.oracle_swiglu_bias.restype = ctypes.c_double
            l.oracle_swiglu_bias.argtypes = [ctypes.c_double] * 4
            l.oracle_e2m1_encode.restype = ctypes.c_uint
            l.oracle_e2m1_encode.argtypes = [ctypes.c_double]
            l.oracle_quant_nvfp4.restype = None
            l.oracle_quant_nvfp4.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p]
            l.oracle_quant_mxfp8.restype = None
            l.oracle_quant_mxfp8.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_void_p, ctypes.c_void_p]
            l.oracle_route_topk.restype = ctypes.c_int
            l.oracle_route_topk.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 4 + [ctypes.c_void_p] * 2
            l.oracle_permute.restype = ctypes.c_int
            l.oracle_permute.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 5 + [ctypes.c_void_p] * 4
            l.oracle_moe_forward.restype = ctypes.c_int
            l.oracle_moe_forward.argtypes = [ctypes.POINTER(_Args), ctypes.c_int, ctypes.c_void_p,
                                             ctypes.c_void_p]
            l.oracle_set_threads.argtypes = [ctypes.c_int]
            l.oracle_get_threads.restype = ctypes.c_int
            _lib = l
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# --- scalar format helpers -------------------------------------------------

def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(code)


def e4m3_value(code: int) -> float:
    return lib().oracle_e4m3_value(code)


def ue8m0_value(b: int) -> float:
    return lib().oracle_ue8m0_value(b)


def bf16_value(h: int) -> float:
    return lib().oracle_bf16_value(h)


def f32_to_bf16(f: float) -> int:
    return lib().oracle_f32_to_bf16(f)


def e4m3_encode(v: float) -> int:
    return lib().oracle_e4m3_encode(v)


def mxfp8_exponent(amax: float) -> int:
    return lib().oracle_mxfp8_exponent(amax)


def situ(g: float, u: float, beta: float, beta_lin: float) -> float:
    return lib().oracle_situ(g, u, beta, beta_lin)


def swiglu_bias(g: float, u: float, alpha: float, beta: float) -> float:
    return float(lib().oracle_swiglu_bias(g, u, alpha, beta))


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def get_threads() -> int:
    return lib().oracle_get_threads()


# --- array entry points ----------------------------------------------------

def e2m1_encode(v: float) -> int:
    return int(lib().oracle_e2m1_encode(float(v)))


def quant_nvfp4(x_bf16_bits: np.ndarray):
    """Per-token NVFP4 quantisation of bf16 rows (uint16 bit patterns [T, H]):
    returns (packed E2M1 uint8 [T, H/2], E4M3 scales uint8 [T, H/16],
    fp32 global scales [T])."""
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    T, H = x.shape
    q = np.zeros((T, H // 2), np.uint8)
    s = np.zeros((T, H // 16), np.uint8)
    g = np.zeros((T,), np.float32)
    lib().oracle_quant_nvfp4(_ptr(x), T, H, _ptr(q), _ptr(s), _ptr(g))
    return q, s, g


def quant_mxfp8(x_bf16_bits: np.ndarray):
    """x: uint16 bf16 bits [T,H] -> (E4M3 uint8 [T,H], UE8M0 uint8 [T,H/32])."""
    x = _c(x_bf16_bits, np.uint16)
    T, H = x.shape
    q = np.empty((T, H), np.uint8)
    s = np.empty((T, H // 32), np.uint8)
    lib().oracle_quant_mxfp8(_ptr(x), T, H, _ptr(q), _ptr(s))
    return q, s


def route_topk(logits: np.ndarray, top_k: int, renormalize: bool = True):
    """Router logits (fp32 [T, E]) -> (int32 ids [T, K] in descending logit
    order, ties to the lower ID; fp32 weights [T, K]: a softmax over the K
    selected logits, or with renormalize=False the selected experts'
    probabilities under a softmax over all E)."""
    x = _c(logits, np.float32)
    T, E = x.shape
    ids = np.empty((T, top_k), np.int32)
    w = np.empty((T, top_k), np.float32)
    if lib().oracle_route_topk(_ptr(x), T, E, int(top_k), 1 if renormalize else 0, _ptr(ids), _ptr(w)) != 0:
        raise ValueError("oracle_route_topk: bad sizes")
    return ids, w


def permute(topk_ids: np.ndarray, num_experts_total: int, num_local_experts: int,
            local_expert_offset: int):
    """Returns (counts, offsets, permuted_src, slot_to_row, R)."""
    ids = _c(topk_ids, np.int32)
    T, K = ids.shape
    E = num_local_experts
    counts = np.empty(max(E, 1), np.int32)
    offsets = np.empty(E + 1, np.int32)
    psrc = np.empty(max(T * K, 1), np.int32)
    s2r = np.empty(max(T * K, 1), np.int32)
    R = lib().oracle_permute(_ptr(ids), T, K, num_experts_total, E, local_expert_offset,
                             _ptr(counts), _ptr(offsets), _ptr(psrc), _ptr(s2r))
    return counts[:E], offsets, psrc[:T * K], s2r[:T * K], R


def moe_forward(*, T, H, I, num_experts_total, num_local_experts, local_expert_offset, top_k,
                act, wt, topk_ids, topk_weights, w1, w1_scale, w2, w2_scale, gemm1_alpha,
                gemm1_beta, hidden_states=None, hidden_states_q=None, hidden_states_scale=None,
                hidden_states_gscale=None, w1_gscale=None, w2_gscale=None, g1_alphas=None,
                g1_alphas_up=None, g2_alphas=None, tokens=None, activation=0,
                apply_topk_in_fc1=0, h1_nvfp4=0) -> np.ndarray:
    """Reference layer output (fp64 [n_tok, H]) for ``tokens`` (all T if None).

    activation: ACT_FN_SITU (gemm1_alpha / gemm1_beta = beta / linear beta)
    or ACT_FN_SWIGLU_BIAS (alpha / beta); apply_topk_in_fc1: the routing
    weight scales H1 (before its rounding) and the un-permute sum is
    unweighted; h1_nvfp4 (NVFP4 weights): H1, rounded to bf16, is requantised
    per token to NVFP4 (the quant_nvfp4 rule) and FC2 takes its exact
    dequantisation.

    hidden_states: uint16 bf16 bits [T,H] (act=ACT_BF16);
    hidden_states_q / hidden_states_scale: E4M3 [T,H] + UE8M0 [T,H/32]
    (ACT_MXFP8) or packed E2M1 [T,H/2] + E4M3 [T,H/16] (ACT_NVFP4) with the
    fp32 per-token hidden_states_gscale [T].
    """
    keep = []

    def c(a, dt):
        a = _c(a, dt)
        keep.append(a)
        return _ptr(a)

    args = _Args(T=T, H=H, I=I, E_total=num_experts_total, E_loc=num_local_experts,
                 off=local_expert_offset, K=top_k, act=act, wt=wt)
    args.x_bf16 = c(hidden_states, np.uint16)
    args.x_q = c(hidden_states_q, np.uint8)
    args.x_s = c(hidden_states_scale, np.uint8)
    args.x_gs = c(hidden_states_gscale, np.float32)
    args.ids = c(topk_ids, np.int32)
    args.wts = c(topk_weights, np.float32)
    args.w1 = c(w1, np.uint8)
    args.w1s = c(w1_scale, np.uint8)
    args.w1_gs = c(w1_gscale, np.float32)
    args.w2 = c(w2, np.uint8)
    args.w2s = c(w2_scale, np.uint8)
    args.w2_gs = c(w2_gscale, np.float32)
    args.beta = c(gemm1_alpha, np.float32)
    args.beta_lin = c(gemm1_beta, np.float32)
    args.alpha_g = c(g1_alphas, np.float32)
    args.alpha_u = c(g1_alphas_up, np.float32)
    args.alpha2 = c(g2_alphas, np.float32)
    args.activation = int(activation)
    args.topk_in_fc1 = int(apply_topk_in_fc1)
    args.h1_nvfp4 = int(h1_nvfp4)
    if tokens is None:
        n_tok, tok_ptr = T, None
    else:
        toks = _c(tokens, np.int32)
        keep.append(toks)
        n_tok, tok_ptr = toks.shape[0], _ptr(toks)
    out = np.empty((max(n_tok, 1), H), np.float64)
    r = lib().oracle_moe_forward(ctypes.byref(args), n_tok, tok_ptr, _ptr(out))
    if r < 0:
        raise ValueError("oracle_moe_forward: bad arguments")
    return out[:n_tok]
