"""DeepSeekMoE layer forward on one B300 (sm_103a): Python binding of libmoe_b300.so.

Argument marshalling only: every step of the layer runs in the library's CUDA kernels,
declared in include/moe.h. Tensors are torch CUDA tensors (PyTorch provides device memory and
streams); the functions take the same arguments as the C entry points of the same name and
raise MoeError on a non-OK status. There is no other implementation behind these names: if
the shared library is missing, importing this package fails.
"""
from __future__ import annotations

import ctypes
import os

__all__ = ["MoeError", "MoeConfig", "MoeWeights", "lib", "make_config", "make_weights",
           "moe_workspace_size", "moe_route", "moe_load_stats", "moe_permute",
           "moe_expert_ffn", "moe_expert_up", "moe_expert_up_gather", "moe_expert_down",
           "moe_combine", "moe_layer_forward", "moe_get_error", "moe_selftest_wait_timeout",
           "moe_status_string", "moe_permute_static_scratch", "moe_stage_timing_start",
           "moe_stage_timing_stop", "moe_bias_update", "moe_seq_balance_loss", "moe_kernel_launches", "moe_group_balance_losses",
           "moe_plan_placement", "MoePlacementConfig", "STAGE_NAMES", "EXPORTED_SYMBOLS", "LIB_PATH", "MOE_OK", "MOE_ERR_INVALID_ARG",
           "MOE_ERR_UNSUPPORTED", "MOE_ERR_WORKSPACE", "MOE_ERR_CUDA", "MOE_ERR_TIMEOUT",
           "MOE_ERR_DEVICE_CHECK"]

# MOE_B300_CHECKED=1 in the environment loads the bounds-checked build (same entry points; the
# kernels check segment offsets, rows and slots and report MOE_ERR_DEVICE_CHECK).
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "libmoe_b300_checked.so" if os.environ.get("MOE_B300_CHECKED") == "1"
                        else "libmoe_b300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, -1, -2, -3
MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_CHECK = -4, -5, -6
MOE_F32, MOE_BF16 = 0, 1
MOE_SOFTMAX, MOE_SIGMOID = 0, 1

EXPORTED_SYMBOLS = ("moe_workspace_size", "moe_route", "moe_load_stats", "moe_permute",
                    "moe_expert_ffn", "moe_expert_up", "moe_expert_down", "moe_combine",
                    "moe_layer_forward", "moe_get_error", "moe_selftest_wait_timeout",
                    "moe_status_string", "moe_last_error_detail", "moe_permute_static_scratch",
                    "moe_stage_timing_start", "moe_stage_timing_stop", "moe_bias_update",
                    "moe_seq_balance_loss", "moe_kernel_launches", "moe_group_balance_losses",
                    "moe_plan_placement", "moe_expert_up_gather")

# Stages of moe_layer_forward as moe_stage_timing_stop reports them (MOE_N_STAGES).
STAGE_NAMES = ("gate", "route", "stats", "permute", "dispatch", "up", "down", "combine")


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({moe_status_string(status)}) {detail}".rstrip())


class MoeConfig(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_routed", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("n_groups", ctypes.c_int32),
                ("topk_groups", ctypes.c_int32), ("group_score_topn", ctypes.c_int32),
                ("score_fn", ctypes.c_int32), ("norm_topk", ctypes.c_int32),
                ("routed_scale", ctypes.c_float), ("capacity_drop", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class MoeWeights(ctypes.Structure):
    _fields_ = [("w_gate", ctypes.c_void_p), ("gate_logit_bias", ctypes.c_void_p),
                ("select_bias", ctypes.c_void_p), ("w13", ctypes.c_void_p),
                ("w2", ctypes.c_void_p), ("w13_shared", ctypes.c_void_p),
                ("w2_shared", ctypes.c_void_p)]


class MoePlacementConfig(ctypes.Structure):
    _fields_ = [("n_experts", ctypes.c_int32), ("n_gpus", ctypes.c_int32),
                ("slots_per_gpu", ctypes.c_int32), ("n_nodes", ctypes.c_int32),
                ("n_groups", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python mixture_experts_routing_sigmoid_b300/build.py`")
    L = ctypes.CDLL(LIB_PATH)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    CFG, W = ctypes.POINTER(MoeConfig), ctypes.POINTER(MoeWeights)
    sig = {
        "moe_workspace_size": (SZ, [CFG, I32]),
        "moe_route": (I32, [CFG, I32, P, W, P, P, P, P, P, SZ, P]),
        "moe_load_stats": (I32, [CFG, I32, P, P, P, P, P, P, P, SZ, P]),
        "moe_permute": (I32, [CFG, I32, P, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_permute_static_scratch": (I32, [CFG, I32, P, P, P, P, P, P, P, P]),
        "moe_expert_ffn": (I32, [CFG, I32, P, P, P, W, P, P, P, SZ, P]),
        "moe_expert_up": (I32, [CFG, I32, P, P, P, W, P, P, P]),
        "moe_expert_up_gather": (I32, [CFG, I32, P, P, P, W, P, P, P]),
        "moe_expert_down": (I32, [CFG, I32, P, P, P, W, P, P, P]),
        "moe_combine": (I32, [CFG, I32, P, P, P, P, P, P]),
        "moe_layer_forward": (I32, [CFG, I32, P, W, P, P, P, P, SZ, P]),
        "moe_get_error": (I32, [P]),
        "moe_selftest_wait_timeout": (I32, [I32, P]),
        "moe_status_string": (ctypes.c_char_p, [I32]),
        "moe_last_error_detail": (ctypes.c_char_p, []),
        "moe_stage_timing_start": (I32, [I32]),
        "moe_bias_update": (I32, [CFG, P, ctypes.c_float, P, P]),
        "moe_seq_balance_loss": (I32, [CFG, I32, I32, P, P, P, P, P, SZ, P]),
        "moe_kernel_launches": (ctypes.c_ulonglong, []),
        "moe_group_balance_losses": (I32, [CFG, I32, P, P, P, P, SZ, P]),
        "moe_plan_placement": (I32, [ctypes.POINTER(MoePlacementConfig), P, P, P, P]),
        "moe_stage_timing_stop": (I32, [P, I32, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype, fn.argtypes = res, args
    return L


lib = _load()


def moe_status_string(status: int) -> str:
    return lib.moe_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where, lib.moe_last_error_detail().decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_config(hidden, n_routed, n_shared, inter, top_k, n_groups=1, topk_groups=1,
                group_score_topn=1, score_fn="softmax", norm_topk=False, routed_scale=1.0,
                capacity_drop=False, dtype="bf16") -> MoeConfig:
    return MoeConfig(hidden=hidden, n_routed=n_routed, n_shared=n_shared, inter=inter,
                     top_k=top_k, n_groups=n_groups, topk_groups=topk_groups,
                     group_score_topn=group_score_topn,
                     score_fn=MOE_SIGMOID if score_fn == "sigmoid" else MOE_SOFTMAX,
                     norm_topk=int(bool(norm_topk)), routed_scale=float(routed_scale),
                     capacity_drop=int(bool(capacity_drop)),
                     dtype=MOE_BF16 if dtype == "bf16" else MOE_F32)


def config_of(layer) -> MoeConfig:
    """moe_config from any object with the LayerConfig attribute names."""
    return make_config(layer.hidden, layer.n_routed, layer.n_shared, layer.inter, layer.top_k,
                       layer.n_groups, layer.topk_groups, layer.group_score_topn,
                       layer.score_fn, layer.norm_topk, layer.routed_scale,
                       layer.capacity_drop, layer.dtype)


def make_weights(w: dict) -> MoeWeights:
    """moe_weights from a dict of CUDA tensors (keys as in the C struct)."""
    return MoeWeights(*[_ptr(w.get(k)) for k, _ in MoeWeights._fields_])


def _cfg(cfg):
    return cfg if isinstance(cfg, MoeConfig) else config_of(cfg)


def _w(w):
    return None if w is None else (w if isinstance(w, MoeWeights) else make_weights(w))


def moe_workspace_size(cfg, T: int) -> int:
    return int(lib.moe_workspace_size(ctypes.byref(_cfg(cfg)), int(T)))


def _ws(ws):
    return (_ptr(ws), 0 if ws is None else ws.numel() * ws.element_size())


def moe_route(cfg, T, x, weights, logits_in, logits_out, topk_idx, topk_w, ws, stream=None):
    p, n = _ws(ws)
    w = _w(weights)
    _check(lib.moe_route(ctypes.byref(_cfg(cfg)), int(T), _ptr(x),
                         None if w is None else ctypes.byref(w), _ptr(logits_in),
                         _ptr(logits_out), _ptr(topk_idx), _ptr(topk_w), p, n,
                         _stream(stream)), "moe_route")


def moe_load_stats(cfg, T, logits, topk_idx, counts, f, P, lb_z, ws, stream=None):
    p, n = _ws(ws)
    _check(lib.moe_load_stats(ctypes.byref(_cfg(cfg)), int(T), _ptr(logits), _ptr(topk_idx),
                              _ptr(counts), _ptr(f), _ptr(P), _ptr(lb_z), p, n,
                              _stream(stream)), "moe_load_stats")


def moe_permute(cfg, T, topk_idx, topk_w, x, offsets, row_token, slot_row, x_perm, ws,
                stream=None, row_w=None):
    """row_w (optional, [T*K] fp32) is a keyword here; the C call takes it after row_token."""
    p, n = _ws(ws)
    _check(lib.moe_permute(ctypes.byref(_cfg(cfg)), int(T), _ptr(topk_idx), _ptr(topk_w),
                           _ptr(x), _ptr(offsets), _ptr(row_token), _ptr(row_w), _ptr(slot_row),
                           _ptr(x_perm), p, n, _stream(stream)), "moe_permute")


def moe_permute_static_scratch(cfg, T, topk_idx, topk_w, x, offsets, row_token, slot_row,
                               x_perm, stream=None):
    """moe_permute for callers that cannot allocate: scratch lives in the library's own
    2.5 MiB device array (T <= 65536; concurrent calls race)."""
    _check(lib.moe_permute_static_scratch(ctypes.byref(_cfg(cfg)), int(T), _ptr(topk_idx),
                                          _ptr(topk_w), _ptr(x), _ptr(offsets), _ptr(row_token),
                                          _ptr(slot_row), _ptr(x_perm), _stream(stream)),
           "moe_permute_static_scratch")


def moe_expert_ffn(cfg, T, x_perm, offsets, x, weights, y_perm, y_shared, ws, stream=None):
    p, n = _ws(ws)
    _check(lib.moe_expert_ffn(ctypes.byref(_cfg(cfg)), int(T), _ptr(x_perm), _ptr(offsets),
                              _ptr(x), ctypes.byref(_w(weights)), _ptr(y_perm), _ptr(y_shared),
                              p, n, _stream(stream)), "moe_expert_ffn")


def moe_expert_up(cfg, T, x_perm, offsets, x, weights, h, h_shared, stream=None):
    _check(lib.moe_expert_up(ctypes.byref(_cfg(cfg)), int(T), _ptr(x_perm), _ptr(offsets),
                             _ptr(x), ctypes.byref(_w(weights)), _ptr(h), _ptr(h_shared),
                             _stream(stream)), "moe_expert_up")


def moe_expert_up_gather(cfg, T, x, row_token, offsets, weights, h, h_shared, stream=None):
    _check(lib.moe_expert_up_gather(ctypes.byref(_cfg(cfg)), int(T), _ptr(x), _ptr(row_token),
                                    _ptr(offsets), ctypes.byref(_w(weights)), _ptr(h),
                                    _ptr(h_shared), _stream(stream)), "moe_expert_up_gather")


def moe_expert_down(cfg, T, h, offsets, h_shared, weights, y_perm, y_shared, stream=None):
    _check(lib.moe_expert_down(ctypes.byref(_cfg(cfg)), int(T), _ptr(h), _ptr(offsets),
                               _ptr(h_shared), ctypes.byref(_w(weights)), _ptr(y_perm),
                               _ptr(y_shared), _stream(stream)), "moe_expert_down")


def moe_combine(cfg, T, y_perm, slot_row, topk_w, y_shared, out, stream=None):
    _check(lib.moe_combine(ctypes.byref(_cfg(cfg)), int(T), _ptr(y_perm), _ptr(slot_row),
                           _ptr(topk_w), _ptr(y_shared), _ptr(out), _stream(stream)),
           "moe_combine")


def moe_layer_forward(cfg, T, x, weights, out, counts, lb_z, ws, stream=None):
    p, n = _ws(ws)
    _check(lib.moe_layer_forward(ctypes.byref(_cfg(cfg)), int(T), _ptr(x),
                                 ctypes.byref(_w(weights)), _ptr(out), _ptr(counts), _ptr(lb_z),
                                 p, n, _stream(stream)), "moe_layer_forward")


def moe_get_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    return int(lib.moe_get_error(_stream(stream)))


def moe_selftest_wait_timeout(timeout_us: int, stream=None):
    _check(lib.moe_selftest_wait_timeout(int(timeout_us), _stream(stream)),
           "moe_selftest_wait_timeout")


def moe_stage_timing_start(max_calls: int):
    _check(lib.moe_stage_timing_start(int(max_calls)), "moe_stage_timing_start")


def moe_stage_timing_stop() -> tuple[dict, int]:
    """-> ({stage name: summed ms over the recorded calls}, number of recorded calls)."""
    ms = (ctypes.c_float * len(STAGE_NAMES))()
    calls = ctypes.c_int32(0)
    _check(lib.moe_stage_timing_stop(ms, len(STAGE_NAMES), ctypes.byref(calls)),
           "moe_stage_timing_stop")
    return dict(zip(STAGE_NAMES, [float(v) for v in ms])), int(calls.value)


def moe_bias_update(cfg, counts, rate: float, select_bias, stream=None):
    _check(lib.moe_bias_update(ctypes.byref(_cfg(cfg)), _ptr(counts), float(rate),
                               _ptr(select_bias), _stream(stream)), "moe_bias_update")


def moe_seq_balance_loss(cfg, T, seq_len, logits, topk_idx, per_seq, loss, ws, stream=None):
    p, n = _ws(ws)
    _check(lib.moe_seq_balance_loss(ctypes.byref(_cfg(cfg)), int(T), int(seq_len), _ptr(logits),
                                    _ptr(topk_idx), _ptr(per_seq), _ptr(loss), p, n,
                                    _stream(stream)), "moe_seq_balance_loss")


def moe_kernel_launches() -> int:
    """Kernels launched by the library so far (a graph-captured launch counts once)."""
    return int(lib.moe_kernel_launches())


def moe_group_balance_losses(cfg, T, logits, topk_idx, losses, ws, stream=None):
    p, n = _ws(ws)
    _check(lib.moe_group_balance_losses(ctypes.byref(_cfg(cfg)), int(T), _ptr(logits),
                                        _ptr(topk_idx), _ptr(losses), p, n, _stream(stream)),
           "moe_group_balance_losses")


def moe_plan_placement(load, n_gpus: int, slots_per_gpu: int, n_nodes: int = 1,
                       n_groups: int = 0):
    """Host-only planner. load: sequence of per-expert loads (int). -> (replicas [N] int32,
    gpu_expert [n_gpus, slots] int32 (-1 = empty), gpu_load [n_gpus] float64) as numpy."""
    import numpy as np
    ld = np.ascontiguousarray(np.asarray(load, dtype=np.int64))
    N = int(ld.size)
    pc = MoePlacementConfig(N, int(n_gpus), int(slots_per_gpu), int(n_nodes), int(n_groups))
    reps = np.zeros(N, np.int32)
    ge = np.zeros((int(n_gpus), int(slots_per_gpu)), np.int32)
    gl = np.zeros(int(n_gpus), np.float64)
    _check(lib.moe_plan_placement(ctypes.byref(pc), ld.ctypes.data, reps.ctypes.data,
                                  ge.ctypes.data, gl.ctypes.data), "moe_plan_placement")
    return reps, ge, gl
