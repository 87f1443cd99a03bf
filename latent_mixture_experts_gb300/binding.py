"""ctypes binding of the lmoe C ABI (include/lmoe.h).

Argument marshalling only: torch supplies device memory and the stream, every
step of the layer runs in the library's CUDA kernels.  The binding fails
loudly when the library is missing or no GPU is present; there is no CPU
path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "liblmoe.so")

LMOE_OK, LMOE_ERR_INVALID_ARG, LMOE_ERR_UNSUPPORTED, LMOE_ERR_CUDA, LMOE_ERR_OOM, LMOE_ERR_TIMEOUT = range(6)
LMOE_ACT_SITU, LMOE_ACT_SWIGLU = 0, 1
LMOE_W_MXFP4, LMOE_W_FP8_BLOCK128 = 0, 1

# Every symbol include/lmoe.h declares.
EXPORTS = ("lmoe_create", "lmoe_route", "lmoe_forward", "lmoe_forward_host", "lmoe_dispatch",
           "lmoe_debug_tensor", "lmoe_sync_status", "lmoe_last_launch_count", "lmoe_set_profiling",
           "lmoe_set_profiling_period",
           "lmoe_profile_get", "lmoe_last_active_experts", "lmoe_destroy", "lmoe_status_string",
           "lmoe_dispatch_noalloc", "lmoe_keep_f32_output", "lmoe_selftest_timeout", "lmoe_tc_peak",
           "lmoe_qb_update", "lmoe_qb_histogram", "lmoe_qb_update_from_histogram",
           "lmoe_ep_dispatch", "lmoe_ep_experts", "lmoe_ep_combine")
NOALLOC_MAX_ASSIGNMENTS = 65536
NOALLOC_MAX_EXPERTS = 2048
PROFILE_ALL_STAGES = 0x1FF
STAGES = ("router", "dispatch", "latent_down", "act_quant", "expert_gate_up", "expert_down", "combine_norm",
          "shared", "output")


class LmoeConfig(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int), ("d_latent", ctypes.c_int), ("n_experts", ctypes.c_int),
                ("top_k", ctypes.c_int), ("d_expert_ff", ctypes.c_int), ("d_shared_ff", ctypes.c_int),
                ("use_latent_norm", ctypes.c_int), ("norm_eps", ctypes.c_float), ("routed_scale", ctypes.c_float),
                ("situ_beta", ctypes.c_float), ("situ_linear_beta", ctypes.c_float), ("act", ctypes.c_int),
                ("expert_wfmt", ctypes.c_int), ("max_tokens", ctypes.c_int), ("act_terms", ctypes.c_int),
                ("act_format", ctypes.c_int), ("ep_size", ctypes.c_int), ("ep_rank", ctypes.c_int),
                ("max_recv_rows", ctypes.c_int)]


_WEIGHT_FIELDS = ("router_w", "router_bias", "w_down_latent", "w_up_latent", "norm_w", "ex_gate_q", "ex_up_q",
                  "ex_down_q", "ex_gate_s", "ex_up_s", "ex_down_s", "sh_gate", "sh_up", "sh_down", "sh_gate_s",
                  "sh_up_s", "sh_down_s")


class LmoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _WEIGHT_FIELDS]


class LmoeError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call} failed: {status_string(status)} ({status})")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH):
    """Load liblmoe.so (built by latent_mixture_experts_gb300.build).  Raises
    if it is absent: nothing here falls back to another implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"lmoe CUDA library not built: {path} missing "
                               "(run python -m latent_mixture_experts_gb300.build)")
        lib = ctypes.CDLL(path)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        sig = {
            "lmoe_create": (I, [ctypes.POINTER(LmoeConfig), ctypes.POINTER(LmoeWeights), P, ctypes.POINTER(P)]),
            "lmoe_route": (I, [P, P, I, P, P, P]),
            "lmoe_forward": (I, [P, P, I, P, P, P, P]),
            "lmoe_forward_host": (I, [P, P, I, P, P]),
            "lmoe_dispatch": (I, [P, P, I, P, P, P, P]),
            "lmoe_debug_tensor": (I, [P, ctypes.c_char_p, P, S, P]),
            "lmoe_sync_status": (I, [P, P]),
            "lmoe_last_launch_count": (I, [P]),
            "lmoe_set_profiling": (I, [P, I, ctypes.c_uint32]),
            "lmoe_set_profiling_period": (I, [P, I]),
            "lmoe_profile_get": (I, [P, I, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(I)]),
            "lmoe_last_active_experts": (I, [P, P]),
            "lmoe_destroy": (I, [P]),
            "lmoe_status_string": (ctypes.c_char_p, [I]),
            "lmoe_dispatch_noalloc": (I, [P, I, I, I, P, P, P, P]),
            "lmoe_keep_f32_output": (I, [P, I]),
            "lmoe_selftest_timeout": (I, [P, ctypes.c_ulonglong, P]),
            "lmoe_tc_peak": (I, [I, I, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double), P]),
            "lmoe_qb_update": (I, [P, P, I, P, P, P]),
            "lmoe_qb_histogram": (I, [P, P, I, P, I, P, P]),
            "lmoe_qb_update_from_histogram": (I, [P, P, I, P, P, P]),
            "lmoe_ep_dispatch": (I, [P, P, I, P, P, P, P, P]),
            "lmoe_ep_experts": (I, [P, P, P, I, P, P]),
            "lmoe_ep_combine": (I, [P, P, I, P, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load_library().lmoe_status_string(int(status)).decode()


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(call: str, st: int):
    if st != LMOE_OK:
        raise LmoeError(call, st)


def lmoe_dispatch_noalloc(topk_idx: torch.Tensor, n_experts: int, counts: torch.Tensor, offsets: torch.Tensor,
                          perm: torch.Tensor, stream=None) -> None:
    """Handle-free dispatch for callers that cannot allocate device memory:
    the caller passes every output buffer (counts int32 [E], offsets int32
    [E+1], perm int32 [T*k]); the library's scratch is a static device array
    (T*k <= 65536, E <= 2048).  Calls that overlap on the GPU race."""
    T, k = topk_idx.shape
    _check("lmoe_dispatch_noalloc", load_library().lmoe_dispatch_noalloc(
        _ptr(topk_idx), T, k, int(n_experts), _ptr(counts), _ptr(offsets), _ptr(perm), _stream(stream)))


TC_KINDS = {"bf16": 0, "e4m3_e4m3": 1, "e2m1_e4m3": 2, "mxfp4": 3, "nvfp4": 4}


def tc_peak(kind: str, iters: int, stream=None) -> float:
    """Measured tensor-pipe rate (TFLOP/s) of one MMA form (include/lmoe_peak.h)."""
    ms, fl = ctypes.c_float(), ctypes.c_double()
    _check("lmoe_tc_peak", load_library().lmoe_tc_peak(TC_KINDS[kind], int(iters), ctypes.byref(ms),
                                                       ctypes.byref(fl), _stream(stream)))
    return fl.value / (ms.value * 1e-3) / 1e12


def make_config(cfg, max_tokens: int, ep_size: int = 1, ep_rank: int = 0, max_recv_rows: int = 0) -> LmoeConfig:
    """C config from an lmoe_inputs.LayerConfig-like object."""
    return LmoeConfig(d_model=cfg.d_model, d_latent=cfg.d_latent, n_experts=cfg.n_experts, top_k=cfg.top_k,
                      d_expert_ff=cfg.d_expert_ff, d_shared_ff=cfg.d_shared_ff,
                      use_latent_norm=int(cfg.use_latent_norm), norm_eps=cfg.norm_eps,
                      routed_scale=cfg.routed_scale, situ_beta=cfg.situ_beta,
                      situ_linear_beta=cfg.situ_linear_beta,
                      act=LMOE_ACT_SITU if cfg.act == "situ" else LMOE_ACT_SWIGLU,
                      expert_wfmt=LMOE_W_MXFP4 if cfg.expert_wfmt == "mxfp4" else LMOE_W_FP8_BLOCK128,
                      max_tokens=int(max_tokens), act_terms=int(getattr(cfg, "act_terms", 2)),
                      act_format=1 if getattr(cfg, "act_format", "e4m3") == "e2m1" else 0,
                      ep_size=int(ep_size), ep_rank=int(ep_rank), max_recv_rows=int(max_recv_rows))


class LatentMoE:
    """One layer instance on the current CUDA device.

    weights: dict of CUDA tensors named as the C weight struct (bf16 tensors
    as torch.bfloat16, codes/scales as torch.uint8, bias float32).  The
    tensors are borrowed: this object keeps references so they outlive the
    handle."""

    def __init__(self, cfg, weights: dict, max_tokens: int, stream=None, ep_size: int = 1, ep_rank: int = 0,
                 max_recv_rows: int = 0):
        lib = load_library()
        if not torch.cuda.is_available():
            raise RuntimeError("lmoe needs a CUDA GPU; no CPU implementation exists")
        self.cfg = cfg
        self.max_tokens = int(max_tokens)
        self._weights = {k: v for k, v in weights.items() if isinstance(v, torch.Tensor)}
        for k, v in self._weights.items():
            if not v.is_cuda or not v.is_contiguous():
                raise ValueError(f"weight {k} must be a contiguous CUDA tensor")
        w = LmoeWeights(**{n: (self._weights[n].data_ptr() if n in self._weights else None)
                           for n in _WEIGHT_FIELDS})
        c = make_config(cfg, max_tokens, ep_size, ep_rank, max_recv_rows)
        self.ep_size = max(1, int(ep_size))
        h = ctypes.c_void_p()
        _check("lmoe_create", lib.lmoe_create(ctypes.byref(c), ctypes.byref(w), _stream(stream), ctypes.byref(h)))
        self._h = h
        self._lib = lib

    # -- calls mirroring the C ABI -------------------------------------
    def lmoe_route(self, x: torch.Tensor, stream=None):
        T = x.shape[0]
        idx = torch.empty(T, self.cfg.top_k, dtype=torch.int32, device=x.device)
        w = torch.empty(T, self.cfg.top_k, dtype=torch.float32, device=x.device)
        _check("lmoe_route", self._lib.lmoe_route(self._h, _ptr(x), T, _ptr(idx), _ptr(w), _stream(stream)))
        return idx, w

    def lmoe_forward(self, x: torch.Tensor, out: torch.Tensor | None = None, return_routing: bool = False,
                     stream=None):
        T = x.shape[0]
        if out is None:
            out = torch.empty(T, self.cfg.d_model, dtype=torch.bfloat16, device=x.device)
        idx = w = None
        if return_routing:
            idx = torch.empty(T, self.cfg.top_k, dtype=torch.int32, device=x.device)
            w = torch.empty(T, self.cfg.top_k, dtype=torch.float32, device=x.device)
        _check("lmoe_forward", self._lib.lmoe_forward(self._h, _ptr(x), T, _ptr(out), _ptr(idx), _ptr(w),
                                                      _stream(stream)))
        return (out, idx, w) if return_routing else out

    def lmoe_forward_host(self, x_host: torch.Tensor, out_host: torch.Tensor, stream=None):
        _check("lmoe_forward_host", self._lib.lmoe_forward_host(self._h, _ptr(x_host), x_host.shape[0],
                                                                _ptr(out_host), _stream(stream)))
        return out_host

    def lmoe_dispatch(self, topk_idx: torch.Tensor, stream=None):
        T = topk_idx.shape[0]
        E = self.cfg.n_experts
        counts = torch.empty(E, dtype=torch.int32, device=topk_idx.device)
        offsets = torch.empty(E + 1, dtype=torch.int32, device=topk_idx.device)
        perm = torch.empty(T * self.cfg.top_k, dtype=torch.int32, device=topk_idx.device)
        _check("lmoe_dispatch", self._lib.lmoe_dispatch(self._h, _ptr(topk_idx), T, _ptr(counts), _ptr(offsets),
                                                        _ptr(perm), _stream(stream)))
        return counts, offsets, perm

    def lmoe_debug_tensor(self, name: str, T: int, stream=None):
        c = self.cfg
        dx = c.d_latent or c.d_model          # width of the expert sum (the latent, or d for K2-style layers)
        shapes = {"logits": ((T, c.n_experts), torch.float32), "xc": ((T, c.d_latent), torch.float32),
                  "u": ((T, dx), torch.float32), "u_hat": ((T, dx), torch.bfloat16),
                  "h_shared": ((T, c.d_shared_ff), torch.bfloat16), "y_shared": ((T, c.d_model), torch.float32),
                  "delta_f32": ((T, c.d_model), torch.float32), "counts": ((c.n_experts,), torch.int32),
                  "x_expert": ((T * c.top_k, dx), torch.float32), "h": ((T * c.top_k, c.d_expert_ff), torch.float32),
                  "offsets": ((c.n_experts + 1,), torch.int32), "perm": ((T * c.top_k,), torch.int32)}
        shape, dt = shapes[name]
        dst = torch.empty(shape, dtype=dt, device="cuda")
        _check("lmoe_debug_tensor", self._lib.lmoe_debug_tensor(self._h, name.encode(), _ptr(dst),
                                                                dst.numel() * dst.element_size(), _stream(stream)))
        return dst

    def lmoe_keep_f32_output(self, enable: bool = True):
        """Keep Delta before its bf16 rounding (debug tensor "delta_f32")."""
        _check("lmoe_keep_f32_output", self._lib.lmoe_keep_f32_output(self._h, int(bool(enable))))

    def lmoe_selftest_timeout(self, limit_ns: int, stream=None):
        """Launch the bounded-wait probe: the next lmoe_sync_status reports a timeout."""
        _check("lmoe_selftest_timeout", self._lib.lmoe_selftest_timeout(self._h, int(limit_ns), _stream(stream)))

    def lmoe_qb_update(self, T: int, logits=None, bias=None, stream=None) -> torch.Tensor:
        """Exact Quantile Balancing update (new biases, fp32 [E]) for a batch
        of T tokens: the given logits [T][E], or the last forward's."""
        nb = torch.empty(self.cfg.n_experts, dtype=torch.float32, device="cuda")
        _check("lmoe_qb_update", self._lib.lmoe_qb_update(self._h, _ptr(logits), int(T), _ptr(bias), _ptr(nb),
                                                          _stream(stream)))
        return nb

    def lmoe_qb_histogram(self, T: int, counts: torch.Tensor, logits=None, bias=None, stream=None):
        """Add a batch's required biases to counts (int32 [E][bins])."""
        _check("lmoe_qb_histogram", self._lib.lmoe_qb_histogram(self._h, _ptr(logits), int(T), _ptr(bias),
                                                                counts.shape[1], _ptr(counts), _stream(stream)))
        return counts

    def lmoe_qb_update_from_histogram(self, counts: torch.Tensor, bias=None, stream=None) -> torch.Tensor:
        nb = torch.empty(self.cfg.n_experts, dtype=torch.float32, device="cuda")
        _check("lmoe_qb_update_from_histogram", self._lib.lmoe_qb_update_from_histogram(
            self._h, _ptr(counts), counts.shape[1], _ptr(bias), _ptr(nb), _stream(stream)))
        return nb

    # -- expert parallelism: the device phases between the caller's exchanges
    def lmoe_ep_dispatch(self, x: torch.Tensor, stream=None):
        """-> (send rows bf16 [T*k][dx] grouped by global expert, expert_counts int32 [E])."""
        c = self.cfg
        T = x.shape[0]
        dx = c.d_latent or c.d_model
        send = torch.empty(T * c.top_k, dx, dtype=torch.bfloat16, device=x.device)
        counts = torch.empty(c.n_experts, dtype=torch.int32, device=x.device)
        _check("lmoe_ep_dispatch", self._lib.lmoe_ep_dispatch(self._h, _ptr(x), T, _ptr(send), _ptr(counts), None,
                                                              None, _stream(stream)))
        return send, counts

    def lmoe_ep_experts(self, recv: torch.Tensor, recv_counts: torch.Tensor, stream=None) -> torch.Tensor:
        """Received rows bf16 [n][dx] and counts int32 [ep_size][E/ep_size] -> expert outputs bf16 [n][dx]."""
        out = torch.empty_like(recv)
        _check("lmoe_ep_experts", self._lib.lmoe_ep_experts(self._h, _ptr(recv), _ptr(recv_counts), recv.shape[0],
                                                            _ptr(out), _stream(stream)))
        return out

    def lmoe_ep_combine(self, ret: torch.Tensor, T: int, stream=None) -> torch.Tensor:
        out = torch.empty(T, self.cfg.d_model, dtype=torch.bfloat16, device=ret.device)
        _check("lmoe_ep_combine", self._lib.lmoe_ep_combine(self._h, _ptr(ret), int(T), _ptr(out), _stream(stream)))
        return out

    def lmoe_sync_status(self, stream=None):
        _check("lmoe_sync_status", self._lib.lmoe_sync_status(self._h, _stream(stream)))

    def lmoe_last_launch_count(self) -> int:
        return int(self._lib.lmoe_last_launch_count(self._h))

    def lmoe_set_profiling(self, reserve_forwards: int, stages=None):
        """Time the named stages (all when None) of the next forwards; an
        empty list or reserve_forwards = 0 with stages=[] turns timing off."""
        if stages is None:
            mask = PROFILE_ALL_STAGES if reserve_forwards else 0
        else:
            mask = 0
            for name in stages:
                mask |= 1 << STAGES.index(name)
        _check("lmoe_set_profiling", self._lib.lmoe_set_profiling(self._h, int(reserve_forwards), mask))

    def lmoe_set_profiling_period(self, every: int):
        """Time only every `every`-th call while profiling is on."""
        _check("lmoe_set_profiling_period", self._lib.lmoe_set_profiling_period(self._h, int(every)))

    def lmoe_profile_get(self) -> dict:
        """{stage name: (summed ms, launches)} since profiling was enabled."""
        out = {}
        for i, name in enumerate(STAGES):
            ms, n = ctypes.c_float(), ctypes.c_int()
            _check("lmoe_profile_get", self._lib.lmoe_profile_get(self._h, i, ctypes.byref(ms), ctypes.byref(n)))
            out[name] = (ms.value, n.value)
        return out

    def lmoe_last_active_experts(self, stream=None) -> int:
        return int(self._lib.lmoe_last_active_experts(self._h, _stream(stream)))

    def lmoe_destroy(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _check("lmoe_destroy", self._lib.lmoe_destroy(self._h))
        self._h = None

    # -- conveniences ----------------------------------------------------
    forward = lmoe_forward
    route = lmoe_route
    dispatch = lmoe_dispatch
    close = lmoe_destroy

    def __del__(self):
        try:
            self.lmoe_destroy()
        except Exception:
            pass
