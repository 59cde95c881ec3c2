"""Python binding of libft (the C ABI in include/ft.h): argument marshalling only.

Every function here has the name of the C entry point without its ``ft_``
prefix and takes plain integers for pointers (device or host addresses, e.g.
``tensor.data_ptr()``) and streams (``torch.cuda.Stream.cuda_stream``).  Every
step of the hot path runs in the CUDA library; there is no Python or CPU
fallback: if libft.so is missing this module raises on first use.

``Context`` is a small convenience owner of an ``ft_ctx*`` that raises
``FtError`` on a non-zero status.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libft.so")

FT_OK = 0
FT_ERR_ARG = -1
FT_ERR_CUDA = -2
FT_ERR_OOM = -3
FT_ERR_CAPACITY = -4
FT_ERR_TIMEOUT = -5
FT_ERR_STATE = -6
FT_ERR_DEVICE = -7
FT_FMT_BF16 = 0
FT_FMT_NVFP4 = 1
FT_FMT_MXFP4 = 2
FT_FMT_FP8 = 3

_c_int = ctypes.c_int32
_c_p = ctypes.c_void_p


class CtlInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("layer", "T", "u", "h", "m", "q0", "q1", "q", "nC", "u_gpu", "n_assign")] + \
               [("clock", ctypes.c_uint32)]


class Counters(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("calls", "unique", "hits", "misses", "fills", "cpu", "assign")]


FT_K_COUNT = 16


class Profile(ctypes.Structure):
    _fields_ = [("ms", ctypes.c_double * FT_K_COUNT), ("launches", ctypes.c_uint64 * FT_K_COUNT)]


# name -> (restype, argtypes)
_SIGS = {
    "ft_abi_version": (_c_int, []),
    "ft_status_str": (ctypes.c_char_p, [_c_int]),
    "ft_record_bytes": (ctypes.c_size_t, [_c_int, _c_int, _c_int]),
    "ft_layer_init": (_c_int, [ctypes.POINTER(_c_p), _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                               _c_int, _c_int, _c_p, _c_p, _c_p, _c_p]),
    "ft_route_ctl": (_c_int, [_c_p, _c_int, _c_int, _c_p, _c_p, _c_p, ctypes.c_double, ctypes.c_double]),
    "ft_moe_forward": (_c_int, [_c_p, _c_p, _c_p, _c_p]),
    "ft_prefill_begin": (_c_int, [_c_p, _c_int]),
    "ft_prefill_layer": (_c_int, [_c_p, _c_int, _c_int, _c_int, _c_int, _c_p, _c_p, _c_p]),
    "ft_cache_resize": (_c_int, [_c_p, _c_int]),
    "ft_measure_link": (_c_int, [_c_p, _c_int, _c_int, ctypes.POINTER(ctypes.c_double)]),
    "ft_get_ctl_state": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p]),
    "ft_set_ctl_state": (_c_int, [_c_p, _c_p, _c_p, _c_p, ctypes.c_uint32]),
    "ft_get_last_ctl": (_c_int, [_c_p, ctypes.POINTER(CtlInfo), _c_p, _c_p, _c_p, _c_p, _c_p, _c_p]),
    "ft_read_slot": (_c_int, [_c_p, _c_int, _c_p]),
    "ft_get_counters": (_c_int, [_c_p, ctypes.POINTER(Counters)]),
    "ft_profile_enable": (_c_int, [_c_p, _c_int]),
    "ft_profile_read": (_c_int, [_c_p, ctypes.POINTER(Profile)]),
    "ft_profile_pause": (_c_int, [_c_p, _c_int]),
    "ft_kernel_name": (ctypes.c_char_p, [_c_int]),
    "ft_num_slots": (_c_int, [_c_p]),
    "ft_expert_ffn_noalloc": (_c_int, [_c_p, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_int, _c_int, _c_int,
                                       _c_p]),
    "ft_noalloc_status": (_c_int, [_c_p]),
    "ft_set_wait_limit": (_c_int, [_c_p, ctypes.c_uint64]),
    "ft_get_status": (_c_int, [_c_p]),
    "ft_destroy": (None, [_c_p]),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load libft.so (built by __graft_entry__.build / build.py); raise if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libft.so is not built ({LIB_PATH}); run moe_expert_cache_gb300/build.py")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class FtError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_str(status)} ({status})")
        self.status = status


def _check(st: int, what: str) -> None:
    if st != FT_OK:
        raise FtError(st, what)


# ---------------------------------------------------------------- raw calls

def abi_version() -> int:
    return load().ft_abi_version()


def status_str(s: int) -> str:
    return load().ft_status_str(s).decode()


def record_bytes(H: int, F: int, fmt: int = FT_FMT_BF16) -> int:
    return load().ft_record_bytes(H, F, fmt)


def layer_init(L, E, k, H, F, S, fmt, T_max, T_prefill_max, host_pool, nvfp4_global, compute_stream,
               transfer_stream):
    h = _c_p()
    st = load().ft_layer_init(ctypes.byref(h), L, E, k, H, F, S, fmt, T_max, T_prefill_max, host_pool,
                              nvfp4_global, compute_stream, transfer_stream)
    return st, h.value


def route_ctl(ctx, layer, T, logits, topk_ids, topk_w, B_P, B_H) -> int:
    return load().ft_route_ctl(ctx, layer, T, logits, topk_ids, topk_w, B_P, B_H)


def moe_forward(ctx, x, partial_C, y) -> int:
    return load().ft_moe_forward(ctx, x, partial_C, y)


def prefill_begin(ctx, layer) -> int:
    return load().ft_prefill_begin(ctx, layer)


def prefill_layer(ctx, buffer, layer, next_layer, T, x, logits, y) -> int:
    return load().ft_prefill_layer(ctx, buffer, layer, next_layer, T, x, logits, y)


def cache_resize(ctx, S_new) -> int:
    return load().ft_cache_resize(ctx, S_new)


def measure_link(ctx, n_records, reps, gbps) -> int:
    return load().ft_measure_link(ctx, n_records, reps, gbps)


def get_ctl_state(ctx, slot_for_id, id_for_slot, stamps, clock) -> int:
    return load().ft_get_ctl_state(ctx, slot_for_id, id_for_slot, stamps, clock)


def set_ctl_state(ctx, slot_for_id, id_for_slot, stamps, clock) -> int:
    return load().ft_set_ctl_state(ctx, slot_for_id, id_for_slot, stamps, clock)


def get_last_ctl(ctx, info, F, C, victims, topk_ids, gates, slots_topk) -> int:
    return load().ft_get_last_ctl(ctx, info, F, C, victims, topk_ids, gates, slots_topk)


def read_slot(ctx, slot, host_dst) -> int:
    return load().ft_read_slot(ctx, slot, host_dst)


def get_counters(ctx, out) -> int:
    return load().ft_get_counters(ctx, out)


def profile_enable(ctx, enable) -> int:
    return load().ft_profile_enable(ctx, enable)


def profile_pause(ctx, paused) -> int:
    return load().ft_profile_pause(ctx, paused)


def profile_read(ctx, out) -> int:
    return load().ft_profile_read(ctx, out)


def kernel_name(kid: int):
    n = load().ft_kernel_name(kid)
    return n.decode() if n else None


def expert_ffn_noalloc(records, n_records, route_records, gates, x, partial_C, y, T, k, H, F, stream=None) -> int:
    """Context-free decode expert FFN that allocates nothing (see include/ft.h)."""
    return load().ft_expert_ffn_noalloc(records, n_records, route_records, gates, x, partial_C, y, T, k, H, F,
                                        stream)


def noalloc_status(stream=None) -> int:
    """Sync `stream`; return and clear the allocation-free path's error word."""
    return load().ft_noalloc_status(stream)


def num_slots(ctx) -> int:
    return load().ft_num_slots(ctx)


def set_wait_limit(ctx, ns) -> int:
    return load().ft_set_wait_limit(ctx, ns)


def get_status(ctx) -> int:
    return load().ft_get_status(ctx)


def destroy(ctx) -> None:
    load().ft_destroy(ctx)


# ------------------------------------------------------------ convenience

def _ptr(a) -> int | None:
    """Address of a numpy array / torch tensor / int; None for None."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if hasattr(a, "data_ptr"):
        return a.data_ptr()
    if hasattr(a, "ctypes"):
        return a.ctypes.data
    raise TypeError(type(a))


class Context:
    """Owner of one ft_ctx*; every method raises FtError on a non-zero status.

    ``host_pool`` is a page-locked host tensor (or address) holding L*E
    records of ``record_bytes(H, F, fmt)`` bytes.  ``fmt`` is FT_FMT_BF16,
    FT_FMT_NVFP4 (then ``nvfp4_global`` is a fp32 array of L*E per-record
    globals), FT_FMT_MXFP4 or FT_FMT_FP8 (block-FP8); the record layouts are
    in include/ft.h.  Streams are ``torch.cuda.Stream.cuda_stream`` handles
    (0: the legacy default stream).
    """

    def __init__(self, L, E, k, H, F, S, host_pool, *, fmt=FT_FMT_BF16, T_max=16, T_prefill_max=0,
                 nvfp4_global=None, compute_stream=0, transfer_stream=0):
        st, h = layer_init(L, E, k, H, F, S, fmt, T_max, T_prefill_max, _ptr(host_pool), _ptr(nvfp4_global),
                           compute_stream or None, transfer_stream or None)
        _check(st, "ft_layer_init")
        self.h = h
        self.L, self.E, self.k, self.H, self.F, self.fmt = L, E, k, H, F, fmt
        self._keep = (host_pool, nvfp4_global)

    def close(self):
        if self.h:
            destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def S(self) -> int:
        return num_slots(self.h)

    def route_ctl(self, layer, T, logits=None, topk_ids=None, topk_w=None, B_P=1.0, B_H=1.0):
        _check(route_ctl(self.h, layer, T, _ptr(logits), _ptr(topk_ids), _ptr(topk_w), B_P, B_H), "ft_route_ctl")

    def moe_forward(self, x, partial_C, y):
        _check(moe_forward(self.h, _ptr(x), _ptr(partial_C), _ptr(y)), "ft_moe_forward")

    def prefill_begin(self, layer):
        _check(prefill_begin(self.h, layer), "ft_prefill_begin")

    def prefill_layer(self, buffer, layer, next_layer, T, x, logits, y):
        _check(prefill_layer(self.h, buffer, layer, next_layer, T, _ptr(x), _ptr(logits), _ptr(y)),
               "ft_prefill_layer")

    def cache_resize(self, S_new):
        _check(cache_resize(self.h, S_new), "ft_cache_resize")

    def measure_link(self, n_records, reps=3):
        """B_P: record-copy GB/s over the host link, measured with the fill path."""
        g = ctypes.c_double(0.0)
        _check(measure_link(self.h, n_records, reps, ctypes.byref(g)), "ft_measure_link")
        return g.value

    def ctl_state(self):
        import numpy as np
        S = self.S
        sfi = np.empty(self.L * self.E, dtype=np.int32)
        ifs = np.empty(S, dtype=np.int32)
        stp = np.empty(S, dtype=np.uint32)
        clk = np.empty(1, dtype=np.uint32)
        _check(get_ctl_state(self.h, _ptr(sfi), _ptr(ifs), _ptr(stp), _ptr(clk)), "ft_get_ctl_state")
        return sfi, ifs, stp, int(clk[0])

    def set_ctl_state(self, slot_for_id, id_for_slot, stamps, clock):
        import numpy as np
        a = np.ascontiguousarray(slot_for_id, dtype=np.int32)
        b = np.ascontiguousarray(id_for_slot, dtype=np.int32)
        c = np.ascontiguousarray(stamps, dtype=np.uint32)
        _check(set_ctl_state(self.h, _ptr(a), _ptr(b), _ptr(c), int(clock)), "ft_set_ctl_state")

    def last_ctl(self, T):
        import numpy as np
        info = CtlInfo()
        E, k = self.E, self.k
        F = np.empty(E, dtype=np.int32)
        C = np.empty(E, dtype=np.int32)
        V = np.empty(E, dtype=np.int32)
        ids = np.empty(T * k, dtype=np.int32)
        g = np.empty(T * k, dtype=np.float32)
        sl = np.empty(T * k, dtype=np.int32)
        _check(get_last_ctl(self.h, ctypes.byref(info), _ptr(F), _ptr(C), _ptr(V), _ptr(ids), _ptr(g), _ptr(sl)),
               "ft_get_last_ctl")
        return {"info": info, "F": F[:info.q].tolist(), "C": C[:info.nC].tolist(), "victims": V[:info.q].tolist(),
                "ids": ids.reshape(T, k), "gates": g.reshape(T, k), "slots_topk": sl.reshape(T, k)}

    def read_slot(self, slot):
        import numpy as np
        out = np.empty(record_bytes(self.H, self.F, self.fmt), dtype=np.uint8)
        _check(read_slot(self.h, slot, _ptr(out)), "ft_read_slot")
        return out

    def counters(self) -> dict:
        c = Counters()
        _check(get_counters(self.h, ctypes.byref(c)), "ft_get_counters")
        return {n: getattr(c, n) for n, _ in Counters._fields_}

    def status(self) -> int:
        return get_status(self.h)

    def set_wait_limit(self, ns: int):
        """Limit of the BF16 decode kernel's progress waits (0: the 2 s default)."""
        _check(set_wait_limit(self.h, ns), "ft_set_wait_limit")

    def profile_enable(self, on: bool = True):
        _check(profile_enable(self.h, 1 if on else 0), "ft_profile_enable")

    def profile_pause(self, paused: bool):
        _check(profile_pause(self.h, 1 if paused else 0), "ft_profile_pause")

    def profile_read(self) -> dict:
        pr = Profile()
        _check(profile_read(self.h, ctypes.byref(pr)), "ft_profile_read")
        out = {}
        for i in range(FT_K_COUNT):
            if pr.launches[i]:
                out[kernel_name(i)] = {"ms": pr.ms[i], "launches": int(pr.launches[i])}
        return out
