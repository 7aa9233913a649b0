"""Python binding of libmegamoe.so, the GB300 fused a8w4 MoE layer forward.

Argument marshalling only: every stage of the layer runs in the library's
sm_103a kernels.  The module-level ``mm_*`` functions are the C entry points
with their C names (see include/megamoe.h); ``MegaMoE`` wraps one handle for
torch tensors.  There is no fallback: if the library is not built, the first
call raises.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

__all__ = ["lib", "MegaMoE", "MegaMoEError", "library_path", "STATUS", "ROUTE_AUTO", "ROUTE_SMALL",
           "ROUTE_LARGE", "ACT_MXFP8", "ACT_BF16", "DUMP_STAGES"]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libmegamoe.so")
# the same library with the device-side bounds checks compiled in (a failed
# check latches MM_ERR_DEVICE with its site instead of indexing out of range)
debug_library_path = os.path.join(_HERE, "libmegamoe_debug.so")

STATUS = {0: "MM_OK", 1: "MM_ERR_INVALID_ARG", 2: "MM_ERR_UNSUPPORTED", 3: "MM_ERR_NOT_READY",
          4: "MM_ERR_CAPACITY", 5: "MM_ERR_CUDA", 6: "MM_ERR_TIMEOUT", 7: "MM_ERR_DEVICE"}
MM_OK, MM_ERR_INVALID_ARG, MM_ERR_UNSUPPORTED, MM_ERR_NOT_READY = 0, 1, 2, 3
MM_ERR_CAPACITY, MM_ERR_CUDA, MM_ERR_TIMEOUT, MM_ERR_DEVICE = 4, 5, 6, 7
ROUTE_AUTO, ROUTE_SMALL, ROUTE_LARGE = 0, 1, 2
ACT_MXFP8, ACT_BF16 = 0, 1          # a8w4 (default), a16w4
# debug stage -> (name, numpy dtype, per-row width: None = flat)
DUMP_STAGES = {0: ("idx", np.int32), 1: ("weights", np.float32), 2: ("phys", np.int32), 3: ("pos", np.int32),
               4: ("offsets", np.int32), 5: ("xq", np.uint8), 6: ("xs", np.uint8), 7: ("hq", np.uint8),
               8: ("hs", np.uint8), 9: ("y", np.uint16), 10: ("info", np.int32),
               11: ("stamps", np.uint64), 12: ("tiles", np.int32)}

_p, _i32, _i64, _sz = C.c_void_p, C.c_int, C.c_int64, C.c_size_t
_SIGS = {
    "mm_create": [_i32, _i32, _i32, _i32, _i32, C.POINTER(_p)],
    "mm_destroy": [_p],
    "mm_set_weights": [_p, _p, _p, _p, _p],
    "mm_set_eplb_map": [_p, _p, _p, _i32],
    "mm_bind_layer": [_p, _i32],
    "mm_set_recording": [_p, _i32],
    "mm_set_route": [_p, _i32],
    "mm_set_activation_format": [_p, _i32],
    "mm_set_shared_experts": [_p, _i32],
    "mm_reserve": [_p, _i64],
    "mm_forward": [_p, _p, _p, _p, _p, _i64, _p],
    "mm_read_counts": [_p, _i32, _p],
    "mm_reset_counts": [_p, _i32],
    "mm_get_status": [_p, C.POINTER(_i32)],
    "mm_debug_dump": [_p, _i32, _p, _sz],
    "mm_debug_size": [_p, _i32, C.POINTER(_sz)],
    "mm_profile_begin": [_p, _i32],
    "mm_profile_end": [_p, _p, _i32, C.POINTER(_i32)],
    "mm_plan_dispatch_static": [_p, _i64, _i32, _p, _p, _p],
    "mm_plan_replicas": [_p, _i32, _i32, _i32, _p, _p],
    "mm_rebalance": [_p, _i32, _i32],
    "mm_set_expert_parallel": [_p, _i32, _i32, _p],
    "mm_ep_reserve": [_p, _i64, _i64],
    "mm_ep_send_rows": [_p, _i64, C.POINTER(_i64)],
    "mm_ep_dispatch": [_p, _p, _p, _p, _i64, _p, _p, _p, _i64, _p, _p],
    "mm_ep_experts": [_p, _p, _p, _p, _i64, _p, _p],
    "mm_ep_combine": [_p, _p, _p, _p],
}
_libs = {}


def lib(debug: bool = False) -> C.CDLL:
    """The loaded library (the bounds-checked build when debug); raises if it
    has not been built."""
    if debug not in _libs:
        path = debug_library_path if debug else library_path
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "moe_layer_serving_gb300.build.build() (needs nvcc, sm_103a)")
        L = C.CDLL(path)
        for name, args in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = C.c_int
        L.mm_status_string.argtypes = [C.c_int]
        L.mm_status_string.restype = C.c_char_p
        _libs[debug] = L
    return _libs[debug]


def _export(name):
    def call(*args):
        return getattr(lib(), name)(*args)
    call.__name__ = name
    call.__doc__ = f"C entry point {name} (include/megamoe.h)."
    return call


for _n in list(_SIGS) + ["mm_status_string"]:
    globals()[_n] = _export(_n)
    __all__.append(_n)


def plan_replicas(load, num_physical: int, max_replicas: int):
    """Host replica planner -> (phys_of_logical int32 [E, R], replica_counts int32 [E])."""
    load = np.ascontiguousarray(load, np.int64)
    E = load.size
    pol = np.zeros((E, max_replicas), np.int32)
    rc = np.zeros(E, np.int32)
    _check(lib().mm_plan_replicas(load.ctypes.data, E, num_physical, max_replicas, pol.ctypes.data, rc.ctypes.data),
           "mm_plan_replicas")
    return pol, rc


class MegaMoEError(RuntimeError):
    def __init__(self, what: str, status: int):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


def _check(st: int, what: str) -> None:
    if st != MM_OK:
        raise MegaMoEError(what, st)


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream  # torch.cuda.Stream


class MegaMoE:
    """One fused MoE layer operator (one handle) on the current CUDA device."""

    def __init__(self, num_experts: int, num_physical: int, topk: int, hidden: int, inter: int,
                 debug: bool = False):
        """E logical and P physical experts, top-k, hidden size H and expert inter size I (mm_create).
        debug: run on the build with device-side bounds checks (libmegamoe_debug.so)."""
        self._lib = lib(debug)
        h = C.c_void_p()
        _check(self._lib.mm_create(num_experts, num_physical, topk, hidden, inter, C.byref(h)), "mm_create")
        self._h = h
        self.E, self.P, self.k, self.H, self.I = num_experts, num_physical, topk, hidden, inter
        self.S = 0

    @property
    def handle(self):
        return self._h

    def close(self) -> None:
        """Free the handle and its device memory (mm_destroy); idempotent."""
        if self._h:
            self._lib.mm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_weights(self, w1, w1_scale, w2, w2_scale) -> None:
        """Device MXFP4 weights of the P physical experts: w1 [P, 2I, H/2] with scales
        [P, 2I, H/32] (gate rows, then up rows), w2 [P, H, I/2] with scales [P, H, I/32];
        copied into the library's tiled layout (mm_set_weights, synchronous)."""
        _check(self._lib.mm_set_weights(self._h, _addr(w1), _addr(w1_scale), _addr(w2), _addr(w2_scale)),
               "mm_set_weights")

    def set_eplb_map(self, phys_of_logical, replica_counts) -> None:
        """Host arrays: physical ids [E, max_replicas] and replica counts [E] (mm_set_eplb_map)."""
        m = np.ascontiguousarray(phys_of_logical, np.int32)
        rc = np.ascontiguousarray(replica_counts, np.int32)
        _check(self._lib.mm_set_eplb_map(self._h, m.ctypes.data, rc.ctypes.data, m.shape[1]), "mm_set_eplb_map")

    def rebalance(self, layer: int, max_replicas: int) -> None:
        """Re-plan the replicas from the counts of `layer` and install them."""
        _check(self._lib.mm_rebalance(self._h, layer, max_replicas), "mm_rebalance")

    def bind_layer(self, layer: int) -> None:
        """Count slot that later forwards record into (mm_bind_layer)."""
        _check(self._lib.mm_bind_layer(self._h, layer), "mm_bind_layer")

    def set_recording(self, on: bool) -> None:
        """Record per-logical-expert token counts in forwards (mm_set_recording)."""
        _check(self._lib.mm_set_recording(self._h, int(bool(on))), "mm_set_recording")

    def set_route(self, route: int) -> None:
        """ROUTE_AUTO, ROUTE_SMALL (fused kernel) or ROUTE_LARGE (multi-launch path)."""
        _check(self._lib.mm_set_route(self._h, route), "mm_set_route")

    def set_activation_format(self, act: int) -> None:
        """ACT_MXFP8 (a8w4) or ACT_BF16 (a16w4); drops the workspace (reserve again)."""
        _check(self._lib.mm_set_activation_format(self._h, act), "mm_set_activation_format")

    def set_shared_experts(self, num_shared: int) -> None:
        """Fused shared experts: every token also goes to physical experts P .. P+S-1
        with weight 1; drops the weights and the workspace (mm_set_shared_experts)."""
        _check(self._lib.mm_set_shared_experts(self._h, num_shared), "mm_set_shared_experts")
        self.S = num_shared

    def set_expert_parallel(self, rank: int, world: int, first=None) -> None:
        """Make this handle rank `rank` of `world` expert-parallel ranks owning physical
        experts [first[rank], first[rank+1]) (default: P split evenly); drops the weights
        and the workspace, after which set_weights takes the rank's own experts only
        (mm_set_expert_parallel)."""
        if first is None:
            first = [(self.P * r) // world for r in range(world + 1)]
        f = np.ascontiguousarray(first, np.int32)
        _check(self._lib.mm_set_expert_parallel(self._h, rank, world, f.ctypes.data), "mm_set_expert_parallel")
        self.ep_rank, self.ep_world, self.ep_first = rank, world, f.copy()

    def ep_reserve(self, max_tokens: int, max_recv_rows: int) -> None:
        """Workspace for dispatching up to max_tokens tokens and receiving up to
        max_recv_rows rows (mm_ep_reserve)."""
        _check(self._lib.mm_ep_reserve(self._h, max_tokens, max_recv_rows), "mm_ep_reserve")

    def ep_send_rows(self, num_tokens: int) -> int:
        """Rows of the send buffers for num_tokens tokens (mm_ep_send_rows)."""
        n = C.c_int64(0)
        _check(self._lib.mm_ep_send_rows(self._h, num_tokens, C.byref(n)), "mm_ep_send_rows")
        return n.value

    def ep_dispatch(self, hidden, logits, bias, send_xq, send_xs, send_eid, num_tokens: int | None = None,
                    stream=None) -> np.ndarray:
        """Route, quantise and pack this rank's tokens into the send buffers; returns the
        row offsets per destination rank, int64 [world + 1] (mm_ep_dispatch, synchronous)."""
        T = hidden.shape[0] if num_tokens is None else num_tokens
        off = np.zeros(self.ep_world + 1, np.int64)
        cap = 0 if send_eid is None else int(send_eid.shape[0])
        if send_xq is not None:
            cap = min(cap, int(send_xq.shape[0]))
        if send_xs is not None:
            cap = min(cap, int(send_xs.shape[0]))
        _check(self._lib.mm_ep_dispatch(self._h, _addr(hidden), _addr(logits), _addr(bias), T, _addr(send_xq),
                                        _addr(send_xs), _addr(send_eid), cap, off.ctypes.data, _stream(stream)),
               "mm_ep_dispatch")
        return off

    def ep_experts(self, recv_xq, recv_xs, recv_eid, y_recv, n: int | None = None, stream=None) -> None:
        """This rank's experts over the received rows -> y_recv in the order received
        (mm_ep_experts)."""
        n = recv_eid.shape[0] if n is None else n
        _check(self._lib.mm_ep_experts(self._h, _addr(recv_xq), _addr(recv_xs), _addr(recv_eid), n, _addr(y_recv),
                                       _stream(stream)), "mm_ep_experts")

    def ep_combine(self, y_back, out, stream=None) -> None:
        """Weighted combine of the returned y rows (send order) into out (mm_ep_combine)."""
        _check(self._lib.mm_ep_combine(self._h, _addr(y_back), _addr(out), _stream(stream)), "mm_ep_combine")

    def reserve(self, max_tokens: int) -> None:
        """Allocate the workspace for up to max_tokens tokens per forward (mm_reserve)."""
        _check(self._lib.mm_reserve(self._h, max_tokens), "mm_reserve")

    def forward(self, hidden, logits, bias, out, num_tokens: int | None = None, stream=None) -> int:
        """Enqueue one forward; returns the status (raises on failure)."""
        T = hidden.shape[0] if num_tokens is None else num_tokens
        st = self._lib.mm_forward(self._h, _addr(hidden), _addr(logits), _addr(bias), _addr(out), T, _stream(stream))
        _check(st, "mm_forward")
        return st

    def read_counts(self, layer: int) -> np.ndarray:
        """int64 counts [E] of slot `layer` (synchronises; mm_read_counts)."""
        out = np.zeros(self.E, np.int64)
        _check(self._lib.mm_read_counts(self._h, layer, out.ctypes.data), "mm_read_counts")
        return out

    def reset_counts(self, layer: int = -1) -> None:
        """Zero slot `layer`'s counts, or every slot's with -1 (mm_reset_counts)."""
        _check(self._lib.mm_reset_counts(self._h, layer), "mm_reset_counts")

    def get_status(self) -> int:
        """Latched device status of earlier forwards (0 = none), cleared by the read (mm_get_status)."""
        code = C.c_int(0)
        _check(self._lib.mm_get_status(self._h, C.byref(code)), "mm_get_status")
        return code.value

    def profile_begin(self, max_launches: int) -> None:
        """Record the dominant kernel's duration for the next max_launches forwards."""
        _check(self._lib.mm_profile_begin(self._h, max_launches), "mm_profile_begin")

    def profile_end(self) -> np.ndarray:
        """Durations (ms) recorded since profile_begin."""
        buf = np.zeros(100000, np.float32)
        n = C.c_int(0)
        _check(self._lib.mm_profile_end(self._h, buf.ctypes.data, buf.size, C.byref(n)), "mm_profile_end")
        return buf[: n.value].copy()

    def last_info(self) -> tuple[int, int, int]:
        """(route taken: 1 small / 2 large, kernels launched, site of the last
        device-side timeout or 0) of the last forward."""
        a = self.debug_dump(10)
        return int(a[0]), int(a[1]), int(a[2])

    def last_gemm(self) -> int:
        """Grouped GEMM kernel of the last forward: 0 none (fused small-input
        kernel), 1 one CTA per unit, 2 CTA pairs (2-SM MMAs), 3 a16w4.  (By
        default the large path launches both a8w4 kernels and the tile scan
        picks one on the device; this names the one that ran.)"""
        return int(self.debug_dump(10)[3])

    def debug_dump(self, stage: int) -> np.ndarray:
        """Intermediate `stage` of the last forward as a flat array (see DUMP_STAGES)."""
        n = C.c_size_t(0)
        _check(self._lib.mm_debug_size(self._h, stage, C.byref(n)), "mm_debug_size")
        dtype = DUMP_STAGES[stage][1]
        buf = np.zeros(n.value // np.dtype(dtype).itemsize, dtype)
        _check(self._lib.mm_debug_dump(self._h, stage, buf.ctypes.data, n.value), "mm_debug_dump")
        return buf
