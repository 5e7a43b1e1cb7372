"""ctypes binding of ``libsitu_moe.so`` (C ABI in ``include/situ_moe.h``).

Argument marshalling only: PyTorch provides device memory and the stream,
every step of the layer runs in the library's CUDA kernels.  There is no
fallback: if the library is not built, or a call returns an error status,
the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

SITU_OK = 0
SITU_ERR_DEVICE_TIMEOUT = 7
SITU_ACT_BF16, SITU_ACT_MXFP8, SITU_ACT_NVFP4 = 0, 1, 2
SITU_ACT_FN_SITU, SITU_ACT_FN_SWIGLU_BIAS = 0, 1
SITU_W_MXFP4, SITU_W_NVFP4 = 0, 1

_lib = None
_lock = threading.Lock()


class SituError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {status_string(status)} (status {status})")
        self.status = status


class SituMoeArgs(ctypes.Structure):
    """Mirror of ``situ_moe_args``."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "T", "H", "I", "num_experts_total", "num_local_experts", "local_expert_offset", "top_k",
        "act_dtype", "weight_dtype")] + [(n, ctypes.c_void_p) for n in (
            "hidden_states", "hidden_states_q", "hidden_states_scale", "hidden_states_gscale",
            "topk_ids", "topk_weights", "w1", "w1_scale", "w1_gscale", "w2", "w2_scale",
            "w2_gscale", "gemm1_alpha", "gemm1_beta", "g1_alphas", "g1_alphas_up", "g2_alphas",
            "out", "scales_packed")] + [(n, ctypes.c_int32) for n in (
                "fuse_combine", "activation", "apply_topk_in_fc1", "h1_nvfp4")] + [("tactic", ctypes.c_int32 * 2)]


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise ImportError(f"{path} is missing: build it with "
                                  "`python -m block_scaled_fp4_permute_gb300.build` "
                                  "(the layer has no CPU fallback)")
            l = ctypes.CDLL(path)
            vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
            l.situ_status_string.restype = ctypes.c_char_p
            l.situ_status_string.argtypes = [ctypes.c_int]
            l.situ_moe_permute_workspace_size.restype = sz
            l.situ_moe_permute_workspace_size.argtypes = [i32, i32, i32]
            l.situ_moe_permute.restype = ctypes.c_int
            l.situ_moe_permute.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
            l.situ_moe_permute_noalloc.restype = ctypes.c_int
            l.situ_moe_permute_noalloc.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp]
            l.situ_moe_route_topk.restype = ctypes.c_int
            l.situ_moe_route_topk.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp]
            l.situ_moe_quant_mxfp8.restype = ctypes.c_int
            l.situ_moe_quant_mxfp8.argtypes = [vp, i32, i32, vp, vp, vp]
            l.situ_moe_quant_nvfp4.restype = ctypes.c_int
            l.situ_moe_quant_nvfp4.argtypes = [vp, i32, i32, vp, vp, vp, vp]
            l.situ_moe_workspace_size.restype = sz
            l.situ_moe_workspace_size.argtypes = [ctypes.POINTER(SituMoeArgs)]
            l.situ_moe_forward.restype = ctypes.c_int
            l.situ_moe_forward.argtypes = [ctypes.POINTER(SituMoeArgs), vp, sz, vp]
            l.situ_moe_forward_profiled.restype = ctypes.c_int
            l.situ_moe_forward_profiled.argtypes = [ctypes.POINTER(SituMoeArgs), vp, sz, vp,
                                                    ctypes.POINTER(ctypes.c_void_p)]
            l.situ_moe_packed_scales_size.restype = sz
            l.situ_moe_packed_scales_size.argtypes = [ctypes.POINTER(SituMoeArgs)]
            l.situ_moe_pack_scales.restype = ctypes.c_int
            l.situ_moe_pack_scales.argtypes = [ctypes.POINTER(SituMoeArgs), vp, sz, vp]
            l.situ_moe_forward_launches.restype = ctypes.c_int32
            l.situ_moe_forward_launches.argtypes = [ctypes.POINTER(SituMoeArgs)]
            l.situ_moe_device_status.restype = ctypes.c_int
            l.situ_moe_device_status.argtypes = [ctypes.POINTER(SituMoeArgs), vp, vp,
                                                 ctypes.POINTER(ctypes.c_int32)]
            l.situ_moe_wait_selftest.restype = ctypes.c_int
            l.situ_moe_wait_selftest.argtypes = [vp, vp]
            l.situ_moe_forward_wait_test.restype = ctypes.c_int
            l.situ_moe_forward_wait_test.argtypes = [ctypes.POINTER(SituMoeArgs), vp, sz, vp, i32, i32]
            l.situ_tc_peak.restype = ctypes.c_int
            l.situ_tc_peak.argtypes = [i32, i32, vp, ctypes.POINTER(ctypes.c_double), vp]
            _lib = l
    return _lib


def status_string(status: int) -> str:
    return lib().situ_status_string(status).decode()


def _check(fn: str, status: int) -> None:
    if status != SITU_OK:
        raise SituError(fn, status)


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ---------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ---------------------------------------------------------------------------

def situ_moe_permute_workspace_size(T: int, top_k: int, num_local_experts: int) -> int:
    return lib().situ_moe_permute_workspace_size(T, top_k, num_local_experts)


def situ_moe_permute(topk_ids: torch.Tensor, num_experts_total: int, num_local_experts: int,
                     local_expert_offset: int, stream=None):
    """Returns (expert_counts, expert_offsets, permuted_src, slot_to_row)."""
    T, K = topk_ids.shape
    dev = topk_ids.device
    counts = torch.empty(num_local_experts, dtype=torch.int32, device=dev)
    offsets = torch.empty(num_local_experts + 1, dtype=torch.int32, device=dev)
    psrc = torch.empty(max(T * K, 1), dtype=torch.int32, device=dev)
    s2r = torch.empty(max(T * K, 1), dtype=torch.int32, device=dev)
    nbytes = situ_moe_permute_workspace_size(T, K, num_local_experts)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    _check("situ_moe_permute", lib().situ_moe_permute(
        _p(topk_ids.contiguous()), T, K, num_experts_total, num_local_experts, local_expert_offset,
        _p(counts), _p(offsets), _p(psrc), _p(s2r), _p(ws), ws.numel(), _stream(stream)))
    return counts, offsets, psrc[:T * K], s2r[:T * K]


def situ_moe_permute_noalloc(topk_ids: torch.Tensor, num_experts_total: int,
                             num_local_experts: int, local_expert_offset: int, out=None,
                             stream=None):
    """situ_moe_permute with the library's fixed scratch instead of a
    workspace.  ``out`` = (counts, offsets, permuted_src, slot_to_row)
    preallocated by the caller; without it they are allocated here with torch
    (the C entry point itself never allocates)."""
    T, K = topk_ids.shape
    dev = topk_ids.device
    if topk_ids.dtype != torch.int32:
        raise TypeError("topk_ids must be int32")
    topk_ids = topk_ids.contiguous()   # a strided view would be read as if packed
    if out is None:
        out = (torch.empty(num_local_experts, dtype=torch.int32, device=dev),
               torch.empty(num_local_experts + 1, dtype=torch.int32, device=dev),
               torch.empty(max(T * K, 1), dtype=torch.int32, device=dev),
               torch.empty(max(T * K, 1), dtype=torch.int32, device=dev))
    counts, offsets, psrc, s2r = out
    # the kernels write every element of these: check what they will be given
    for t, n, what in ((counts, num_local_experts, "expert_counts"),
                       (offsets, num_local_experts + 1, "expert_offsets"),
                       (psrc, T * K, "permuted_src"), (s2r, T * K, "slot_to_row")):
        if t.dtype != torch.int32 or t.device != dev or not t.is_contiguous() or t.numel() < n:
            raise ValueError(f"{what}: needs a contiguous int32 tensor of >= {n} elements on {dev}")
    _check("situ_moe_permute_noalloc", lib().situ_moe_permute_noalloc(
        _p(topk_ids), T, K, num_experts_total, num_local_experts, local_expert_offset,
        _p(counts), _p(offsets), _p(psrc), _p(s2r), _stream(stream)))
    return counts, offsets, psrc[:T * K], s2r[:T * K]


def situ_moe_route_topk(router_logits: torch.Tensor, top_k: int, renormalize: bool = True, stream=None,
                        out=None):
    """Router logits fp32 [T, E] -> (int32 topk_ids [T, K], fp32 topk_weights
    [T, K]): the K largest logits (ties to the lower ID) and a softmax over
    them (renormalize) or their softmax probabilities over all E."""
    if router_logits.dtype != torch.float32:
        raise TypeError("router_logits must be fp32")
    logits = router_logits.contiguous()
    T, E = logits.shape
    if out is None:
        ids = torch.empty((T, top_k), dtype=torch.int32, device=logits.device)
        w = torch.empty((T, top_k), dtype=torch.float32, device=logits.device)
    else:
        ids, w = out
    _check("situ_moe_route_topk", lib().situ_moe_route_topk(
        _p(logits), T, E, int(top_k), 1 if renormalize else 0, _p(ids), _p(w), _stream(stream)))
    return ids, w


def situ_moe_quant_mxfp8(x_bf16: torch.Tensor, stream=None, out=None):
    """bf16 [T,H] -> (E4M3 uint8 [T,H], UE8M0 uint8 [T,H/32])."""
    T, H = x_bf16.shape
    if out is None:
        q = torch.empty((T, H), dtype=torch.uint8, device=x_bf16.device)
        s = torch.empty((T, H // 32), dtype=torch.uint8, device=x_bf16.device)
    else:
        q, s = out
    _check("situ_moe_quant_mxfp8", lib().situ_moe_quant_mxfp8(
        _p(x_bf16), T, H, _p(q), _p(s), _stream(stream)))
    return q, s


def situ_moe_quant_nvfp4(x_bf16: torch.Tensor, stream=None, out=None):
    """bf16 [T,H] -> (packed E2M1 uint8 [T,H/2], E4M3 uint8 [T,H/16], fp32 [T])."""
    T, H = x_bf16.shape
    if out is None:
        q = torch.empty((T, H // 2), dtype=torch.uint8, device=x_bf16.device)
        s = torch.empty((T, H // 16), dtype=torch.uint8, device=x_bf16.device)
        g = torch.empty((T,), dtype=torch.float32, device=x_bf16.device)
    else:
        q, s, g = out
    _check("situ_moe_quant_nvfp4", lib().situ_moe_quant_nvfp4(
        _p(x_bf16), T, H, _p(q), _p(s), _p(g), _stream(stream)))
    return q, s, g


def make_args(*, T, H, I, num_experts_total, num_local_experts, local_expert_offset, top_k,
              act_dtype, weight_dtype, topk_ids, topk_weights, w1, w1_scale, w2, w2_scale,
              gemm1_alpha, gemm1_beta, out, hidden_states=None, hidden_states_q=None,
              hidden_states_scale=None, hidden_states_gscale=None, w1_gscale=None, w2_gscale=None,
              g1_alphas=None, g1_alphas_up=None, g2_alphas=None) -> SituMoeArgs:
    a = SituMoeArgs(T=T, H=H, I=I, num_experts_total=num_experts_total,
                    num_local_experts=num_local_experts, local_expert_offset=local_expert_offset,
                    top_k=top_k, act_dtype=act_dtype, weight_dtype=weight_dtype)
    a.tactic[0] = a.tactic[1] = -1   # auto
    for name, t in dict(hidden_states=hidden_states, hidden_states_q=hidden_states_q,
                        hidden_states_scale=hidden_states_scale,
                        hidden_states_gscale=hidden_states_gscale, topk_ids=topk_ids,
                        topk_weights=topk_weights, w1=w1, w1_scale=w1_scale, w1_gscale=w1_gscale,
                        w2=w2, w2_scale=w2_scale, w2_gscale=w2_gscale, gemm1_alpha=gemm1_alpha,
                        gemm1_beta=gemm1_beta, g1_alphas=g1_alphas, g1_alphas_up=g1_alphas_up,
                        g2_alphas=g2_alphas, out=out).items():
        setattr(a, name, None if t is None else t.data_ptr())
    return a


def situ_moe_workspace_size(args: SituMoeArgs) -> int:
    return lib().situ_moe_workspace_size(ctypes.byref(args))


def situ_moe_packed_scales_size(args: SituMoeArgs) -> int:
    return lib().situ_moe_packed_scales_size(ctypes.byref(args))


def situ_moe_pack_scales(args: SituMoeArgs, packed: torch.Tensor, stream=None) -> None:
    """Packs the weight scales of ``args`` into ``packed`` (uint8 device
    tensor of at least situ_moe_packed_scales_size bytes)."""
    _check("situ_moe_pack_scales", lib().situ_moe_pack_scales(
        ctypes.byref(args), _p(packed), packed.numel() * packed.element_size(), _stream(stream)))


def situ_moe_forward_launches(args: SituMoeArgs) -> int:
    """Kernels situ_moe_forward enqueues for ``args`` (-1: invalid)."""
    return lib().situ_moe_forward_launches(ctypes.byref(args))


def situ_moe_forward(args: SituMoeArgs, workspace: torch.Tensor, stream=None) -> None:
    _check("situ_moe_forward", lib().situ_moe_forward(
        ctypes.byref(args), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


SITU_SELFTEST_WAIT_CODE = 99   # include/situ_moe.h


def situ_moe_wait_selftest(status: torch.Tensor, stream=None) -> None:
    """One bounded device wait made to run out (the failure path): after the
    wait limit the kernel records SITU_SELFTEST_WAIT_CODE in ``status`` (an
    int32 tensor on the device, zeroed by the caller) and returns."""
    _check("situ_moe_wait_selftest", lib().situ_moe_wait_selftest(_p(status), _stream(stream)))


def situ_moe_forward_wait_test(args: SituMoeArgs, workspace: torch.Tensor, skip_stage: int, wait_us: int,
                               stream=None) -> None:
    """situ_moe_forward whose FC1 (block-scaled decode tiles) leaves K stage
    ``skip_stage`` of CTA 0 unissued, with every wait limited to ``wait_us``:
    the failure path on purpose (read the outcome with situ_moe_device_status)."""
    _check("situ_moe_forward_wait_test", lib().situ_moe_forward_wait_test(
        ctypes.byref(args), _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream),
        int(skip_stage), int(wait_us)))


SITU_TC_MXF8F6F4, SITU_TC_MXF4NVF4, SITU_TC_BF16 = 0, 1, 2
TC_KIND_NAMES = {SITU_TC_MXF8F6F4: "mxf8f6f4", SITU_TC_MXF4NVF4: "mxf4nvf4", SITU_TC_BF16: "bf16"}


def situ_tc_peak(kind: int, mmas_per_sm: int, status: torch.Tensor, stream=None) -> float:
    """Enqueues the MMA-throughput kernel of ``kind`` (SITU_TC_*) with
    ``mmas_per_sm`` MMAs per SM; returns the launch's dense FLOPs.  ``status``
    is an int32 device tensor zeroed by the caller (98 after a timed-out wait)."""
    flops = ctypes.c_double(0.0)
    _check("situ_tc_peak", lib().situ_tc_peak(int(kind), int(mmas_per_sm), _p(status),
                                              ctypes.byref(flops), _stream(stream)))
    return float(flops.value)


def situ_moe_device_status(args: SituMoeArgs, workspace: torch.Tensor, stream=None) -> int:
    """Waits for ``stream`` and returns the device status word of the last
    forward run with this workspace: 0, or the code of the first bounded
    wait a kernel gave up (the C call's SITU_ERR_DEVICE_TIMEOUT is not
    raised, it is reported through the code)."""
    code = ctypes.c_int32(0)
    st = lib().situ_moe_device_status(ctypes.byref(args), _p(workspace), _stream(stream),
                                      ctypes.byref(code))
    if st not in (0, SITU_ERR_DEVICE_TIMEOUT):
        _check("situ_moe_device_status", st)
    return int(code.value)


PROFILE_STAGES = ("permute", "gather", "fc1", "fc2", "combine")


def situ_moe_forward_profiled(args: SituMoeArgs, workspace: torch.Tensor, events, stream=None):
    """situ_moe_forward recording ``events`` (len(PROFILE_STAGES) + 1
    torch.cuda.Event objects with timing enabled) around each stage."""
    assert len(events) == len(PROFILE_STAGES) + 1
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check("situ_moe_forward_profiled", lib().situ_moe_forward_profiled(
        ctypes.byref(args), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream), arr))


class Layer:
    """Keeps the argument struct and a workspace for one workload, so that a
    forward call is a single C-ABI call (the bench times exactly this)."""

    def __init__(self, wl, out: Optional[torch.Tensor] = None, x_q=None, x_scale=None,
                 pack_scales: bool = True, fuse_combine: bool = False, activation: int = 0,
                 apply_topk_in_fc1: bool = False, h1_nvfp4: bool = False):
        self.wl = wl
        dev = wl.x_bf16.device
        self.out = out if out is not None else torch.empty((wl.T, wl.H), dtype=torch.bfloat16,
                                                           device=dev)
        kw = dict(T=wl.T, H=wl.H, I=wl.I, num_experts_total=wl.E_total,
                  num_local_experts=wl.E_loc, local_expert_offset=wl.off, top_k=wl.K,
                  act_dtype=wl.act, weight_dtype=wl.wt, topk_ids=wl.topk_ids,
                  topk_weights=wl.topk_weights, w1=wl.w1, w1_scale=wl.w1_scale, w2=wl.w2,
                  w2_scale=wl.w2_scale, gemm1_alpha=wl.gemm1_alpha, gemm1_beta=wl.gemm1_beta,
                  g1_alphas=wl.g1_alphas, g1_alphas_up=wl.g1_alphas_up, g2_alphas=wl.g2_alphas,
                  w1_gscale=wl.w1_gscale, w2_gscale=wl.w2_gscale, out=self.out)
        if wl.act == SITU_ACT_BF16:
            kw["hidden_states"] = wl.x_bf16
        elif wl.act == SITU_ACT_MXFP8:
            if x_q is None:
                x_q = torch.empty((wl.T, wl.H), dtype=torch.uint8, device=dev)
                x_scale = torch.empty((wl.T, wl.H // 32), dtype=torch.uint8, device=dev)
            self.x_q, self.x_scale = x_q, x_scale
            kw["hidden_states_q"], kw["hidden_states_scale"] = x_q, x_scale
        else:
            # NVFP4: quantised from the bf16 hidden states on the GPU in every call
            self.x_q = torch.empty((wl.T, wl.H // 2), dtype=torch.uint8, device=dev)
            self.x_scale = torch.empty((wl.T, wl.H // 16), dtype=torch.uint8, device=dev)
            self.x_gscale = torch.empty((wl.T,), dtype=torch.float32, device=dev)
            kw["hidden_states_q"], kw["hidden_states_scale"] = self.x_q, self.x_scale
            kw["hidden_states_gscale"] = self.x_gscale
        self._keep = kw
        self.args = make_args(**kw)
        self.args.fuse_combine = 1 if fuse_combine else 0
        self.args.activation = int(activation)
        self.args.apply_topk_in_fc1 = 1 if apply_topk_in_fc1 else 0
        self.args.h1_nvfp4 = 1 if h1_nvfp4 else 0
        # weight scales in the block-scaled GEMMs' layout, packed once per
        # weight set (as at weight-load time) when the shapes use it
        self.scales_packed = None
        np_ = situ_moe_packed_scales_size(self.args) if pack_scales else 0
        if np_ > 0:
            self.scales_packed = torch.empty(np_, dtype=torch.uint8, device=dev)
            situ_moe_pack_scales(self.args, self.scales_packed)
            self.args.scales_packed = self.scales_packed.data_ptr()
        n = situ_moe_workspace_size(self.args)
        self.workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)

    def launches(self) -> int:
        """Kernels one __call__ enqueues (the forward, plus the activation
        quantisation for MXFP8 and NVFP4 activations)."""
        return situ_moe_forward_launches(self.args) + (0 if self.wl.act == SITU_ACT_BF16 else 1)

    def _quant(self, stream):
        if self.wl.act == SITU_ACT_MXFP8:
            situ_moe_quant_mxfp8(self.wl.x_bf16, stream, out=(self.x_q, self.x_scale))
        elif self.wl.act == SITU_ACT_NVFP4:
            situ_moe_quant_nvfp4(self.wl.x_bf16, stream, out=(self.x_q, self.x_scale, self.x_gscale))

    def device_status(self, stream=None) -> int:
        """0 when every bounded device wait of the last call completed."""
        return situ_moe_device_status(self.args, self.workspace, stream)

    def profiled(self, events, quant_events=None, stream=None) -> torch.Tensor:
        """Like __call__, recording per-stage events (see situ_moe_forward_profiled);
        ``quant_events`` (start, end) bracket the activation quantisation."""
        if self.wl.act != SITU_ACT_BF16:
            if quant_events:
                quant_events[0].record(stream)
            self._quant(stream)
            if quant_events:
                quant_events[1].record(stream)
        situ_moe_forward_profiled(self.args, self.workspace, events, stream)
        return self.out

    def capture(self, warmup: bool = True):
        """A CUDA graph of one __call__ (the activation quantisation, if any,
        and the forward's kernels, with their programmatic dependencies).
        situ_moe_forward never synchronises the host, so a call can be
        captured; the graph replays on the same buffers.  Returns the
        torch.cuda.CUDAGraph; ``graph.replay()`` runs one layer pass."""
        if warmup:   # one eager call first: per-device attribute set-up
            self()
            torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                self(stream=s)
        torch.cuda.current_stream().wait_stream(s)
        return g

    def __call__(self, stream=None) -> torch.Tensor:
        """One pass of the layer; for MXFP8 and NVFP4 activations this includes
        their quantisation from the bf16 hidden states."""
        self._quant(stream)
        situ_moe_forward(self.args, self.workspace, stream)
        return self.out
