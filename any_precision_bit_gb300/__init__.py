"""Python binding of libpw.so (include/pw.h): argument marshalling only.

Every function keeps its C name and signature; device buffers are passed as torch
tensors (or raw integer addresses), host buffers as numpy arrays.  A call that returns
a status other than PW_OK raises ``PwError`` with ``pw_last_error``'s message.  There is
no fallback: if libpw.so has not been built, importing works but the first call raises.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpw.so")

PW_OK, PW_ERR_INVALID, PW_ERR_CUDA, PW_ERR_OOM, PW_ERR_STATE, PW_ERR_TIMEOUT, PW_ERR_BUSY, PW_ERR_RANGE = range(8)
PW_FLAG_POISON = 1
PW_ACCUMULATE = 1
PW_PRENORM = 2
PW_PAGE_GPU, PW_PAGE_CPU, PW_PAGE_TO_CPU, PW_PAGE_TO_GPU = range(4)
STATUS_NAMES = {0: "PW_OK", 1: "PW_ERR_INVALID", 2: "PW_ERR_CUDA", 3: "PW_ERR_OOM",
                4: "PW_ERR_STATE", 5: "PW_ERR_TIMEOUT", 6: "PW_ERR_BUSY",
                7: "PW_ERR_RANGE"}


class PwError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class pw_desc(C.Structure):
    _fields_ = [("L", C.c_int), ("E", C.c_int), ("H", C.c_int), ("I", C.c_int), ("K", C.c_int),
                ("Is", C.c_int), ("bmax", C.c_int), ("bits_mask", C.c_uint32), ("renorm", C.c_int),
                ("device", C.c_int), ("max_tokens", C.c_int), ("flags", C.c_int)]


class pw_block_info(C.Structure):
    _fields_ = [("layer", C.c_int), ("expert", C.c_int), ("u", C.c_int), ("N", C.c_int), ("K", C.c_int),
                ("q", C.c_int), ("d", C.c_int), ("pending_q", C.c_int), ("state", C.c_int * 8),
                ("M", C.c_int64 * 9)]


class pw_mem_info(C.Structure):
    _fields_ = [("resident_bytes", C.c_int64), ("device_pool_bytes", C.c_int64),
                ("device_pool_free", C.c_int64), ("pinned_bytes", C.c_int64), ("scratch_bytes", C.c_int64),
                ("held_bytes", C.c_int64)]


class pw_kv_stats(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("budget_bytes", "block_bytes", "weight_bytes", "capacity_blocks",
                                         "used_blocks", "pending_blocks", "free_blocks", "headroom_bytes")]


class pw_obs(C.Structure):
    _fields_ = [("T_blk", C.c_int), ("F_blk", C.c_int), ("B_KV", C.c_double), ("R", C.c_int),
                ("mass", C.c_void_p), ("phi", C.c_void_p), ("rho_hat", C.c_void_p)]


class pw_request_signals(C.Structure):
    _fields_ = [("mass", C.c_void_p), ("rho_hat", C.c_void_p), ("conf", C.c_void_p), ("rho_min", C.c_double),
                ("rho_max", C.c_double), ("kv_blocks", C.c_double)]


class pw_offline(C.Structure):
    _fields_ = [("n_bits", C.c_int), ("s", C.c_void_p), ("head_w", C.c_void_p), ("head_a", C.c_void_p),
                ("head_c", C.c_void_p), ("alpha", C.c_double), ("rho_min", C.c_double),
                ("rho_max", C.c_double), ("eps", C.c_double), ("n_buckets", C.c_int), ("mu", C.c_void_p),
                ("floors", C.c_void_p), ("n_stages", C.c_int)]


class pw_plan_entry(C.Structure):
    _fields_ = [("block", C.c_int), ("from_bits", C.c_int), ("to_bits", C.c_int), ("delta", C.c_double)]


class pw_plan(C.Structure):
    _fields_ = [("entries", C.POINTER(pw_plan_entry)), ("capacity", C.c_int), ("n", C.c_int),
                ("kind", C.c_int), ("stage", C.c_int), ("D", C.c_double), ("total", C.c_double)]


class pw_plan_problem(C.Structure):
    _fields_ = [("n_blocks", C.c_int), ("n_bits", C.c_int), ("L", C.c_int), ("E", C.c_int),
                ("bits", C.c_void_p), ("q", C.c_void_p), ("q_init", C.c_void_p), ("utype", C.c_void_p),
                ("layer", C.c_void_p), ("expert", C.c_void_p), ("M", C.c_void_p)]


_P = C.c_void_p
_I = C.c_int
_SIGS = {
    "pw_create": [C.POINTER(pw_desc), C.POINTER(_P)],
    "pw_destroy": [_P],
    "pw_last_error": [_P],
    "pw_version": [],
    "pw_set_stream": [_P, _P],
    "pw_get_stream": [_P, C.POINTER(_P)],
    "pw_pack": [_P, _I, _I, _I, _P, _P, _I],
    "pw_set_router": [_P, _I, _P, _P],
    "pw_set_shared": [_P, _I, _P, _P],
    "pw_set_shared_gate": [_P, _I, _P],
    "pw_routing_features": [_P, _I, _P, _I],
    "pw_moe_forward": [_P, _I, _P, _I, _P, _P, _P, _I, _P],
    "pw_check": [_P],
    "pw_stack_forward": [_P, _P, _I, _P],
    "pw_stack_forward_host": [_P, _P, _I, _P],
    "pw_routing_stats": [_P, _I, _P, _P, _I],
    "pw_set_bits": [_P, _I, _I],
    "pw_offload": [_P, _I, _I],
    "pw_reload": [_P, _I, _I],
    "pw_commit": [_P, C.POINTER(_I)],
    "pw_sync_io": [_P],
    "pw_query": [_P, _I, C.POINTER(pw_block_info)],
    "pw_memory": [_P, C.POINTER(pw_mem_info)],
    "pw_set_fault": [_P, _I, _I],
    "pw_plan_host": [C.POINTER(pw_plan_problem), C.POINTER(pw_obs), C.POINTER(pw_offline), C.POINTER(pw_plan)],
    "pw_plan_step": [_P, C.POINTER(pw_obs), C.POINTER(pw_offline), C.POINTER(pw_plan)],
    "pw_merge_requests": [C.POINTER(pw_request_signals), _I, _I, _I, _I, _I, _P, _P, _P, C.POINTER(C.c_double),
                          C.POINTER(C.c_double)],
    "pw_route_noalloc": [_P, _I, _P, _I, _P, _P, _I, _P],
    "pw_kv_create": [C.c_int64, C.c_int64, C.POINTER(C.c_void_p)],
    "pw_kv_destroy": [_P],
    "pw_kv_set_weight_bytes": [_P, C.c_int64],
    "pw_kv_attach": [_P, _P],
    "pw_kv_announce": [_P, C.c_int64, C.c_int64],
    "pw_kv_grow": [_P, C.c_int64, C.c_int64, _P],
    "pw_kv_release": [_P, C.c_int64, C.POINTER(C.c_int64)],
    "pw_kv_request": [_P, C.c_int64, C.POINTER(C.c_int64), C.POINTER(C.c_int64)],
    "pw_kv_blocks": [_P, C.c_int64, _P, C.c_int64, C.POINTER(C.c_int64)],
    "pw_kv_get_stats": [_P, C.POINTER(pw_kv_stats)],
    "pw_set_profiling": [_P, _I],
    "pw_set_gemv_tokens": [_P, _I],
    "pw_profile_read": [_P, _I, _P],
    "pw_tc_selftest": [_P, _P, _I, _I, _I, _P, _P, _P],
    "pw_unpack_indices": [_P, _I, _I, _P],
    "pw_dequant": [_P, _I, _I, _P],
    "pw_pack_planes_host": [_P, _I, _I, _I, _P],
    "pw_tile_planes_host": [_P, _I, _I, _I, _I, _P],
    "pw_untile_planes_host": [_P, _I, _I, _I, _I, _P],
}

_lib = None


def lib():
    """The loaded libpw.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libpw.so is not built; run any_precision_bit_gb300._build.build()")
        L = C.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = None if name in ("pw_destroy", "pw_kv_destroy") else (C.c_char_p if name in ("pw_last_error", "pw_version") else C.c_int)
        _lib = L
    return _lib


def _ptr(obj):
    """Address of a torch tensor, numpy array, integer address or None."""
    if obj is None:
        return None
    if isinstance(obj, int):
        return obj
    if isinstance(obj, np.ndarray):
        if not obj.flags["C_CONTIGUOUS"]:
            raise ValueError("numpy arrays must be C-contiguous")
        return obj.ctypes.data
    if hasattr(obj, "data_ptr"):
        if hasattr(obj, "is_contiguous") and not obj.is_contiguous():
            raise ValueError("tensors must be contiguous")
        return obj.data_ptr()
    if hasattr(obj, "cuda_stream"):
        return obj.cuda_stream
    raise TypeError(f"cannot take the address of {type(obj)}")


def _check(st, ctx=None):
    if st != PW_OK:
        msg = lib().pw_last_error(ctx)
        raise PwError(st, msg.decode() if msg else "")
    return st


def _stream(s):
    if s is None:
        return None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s)


# ------------------------------------------------------------------ the ABI, one to one
def pw_version():
    return lib().pw_version().decode()


def pw_create(desc: pw_desc):
    h = C.c_void_p()
    _check(lib().pw_create(C.byref(desc), C.byref(h)))
    return h.value


def pw_destroy(ctx):
    lib().pw_destroy(ctx)


def pw_last_error(ctx=None):
    return lib().pw_last_error(ctx).decode()


def pw_set_stream(ctx, stream):
    _check(lib().pw_set_stream(ctx, _stream(stream)), ctx)


def pw_get_stream(ctx):
    s = C.c_void_p()
    _check(lib().pw_get_stream(ctx, C.byref(s)), ctx)
    return s.value or 0


def pw_pack(ctx, layer, expert, u, idx, lut, q_init):
    _check(lib().pw_pack(ctx, layer, expert, u, _ptr(idx), _ptr(lut), q_init), ctx)


def pw_set_router(ctx, layer, Wr, bias=None):
    _check(lib().pw_set_router(ctx, layer, _ptr(Wr), _ptr(bias)), ctx)


def pw_set_shared(ctx, layer, wgu, wd):
    _check(lib().pw_set_shared(ctx, layer, _ptr(wgu), _ptr(wd)), ctx)


def pw_set_shared_gate(ctx, layer, wsg=None):
    if wsg is not None and not hasattr(wsg, "data_ptr"):
        wsg = np.ascontiguousarray(wsg, dtype=np.float32)
    _check(lib().pw_set_shared_gate(ctx, layer, _ptr(wsg)), ctx)


def pw_moe_forward(ctx, layer, x, T, y, ids=None, w=None, flags=0, stream=None):
    _check(lib().pw_moe_forward(ctx, layer, _ptr(x), T, _ptr(y), _ptr(ids), _ptr(w), flags, _stream(stream)), ctx)


def pw_check(ctx):
    _check(lib().pw_check(ctx), ctx)


def pw_stack_forward(ctx, x, T, stream=None):
    _check(lib().pw_stack_forward(ctx, _ptr(x), T, _stream(stream)), ctx)


def pw_stack_forward_host(ctx, x_host, T, y_host):
    _check(lib().pw_stack_forward_host(ctx, _ptr(x_host), T, _ptr(y_host)), ctx)


def pw_routing_stats(ctx, layer, E, reset=False):
    cnt = np.zeros(E, dtype=np.float64)
    ws = np.zeros(E, dtype=np.float64)
    _check(lib().pw_routing_stats(ctx, layer, _ptr(cnt), _ptr(ws), int(reset)), ctx)
    return cnt, ws


def pw_routing_features(ctx, layer, E, reset=False):
    phi = np.zeros((E, 3), dtype=np.float64)
    _check(lib().pw_routing_features(ctx, layer, _ptr(phi), int(reset)), ctx)
    return phi


def pw_set_bits(ctx, block, q):
    _check(lib().pw_set_bits(ctx, block, q), ctx)


def pw_offload(ctx, block, q_new):
    _check(lib().pw_offload(ctx, block, q_new), ctx)


def pw_reload(ctx, block, q_new):
    _check(lib().pw_reload(ctx, block, q_new), ctx)


def pw_commit(ctx):
    n = C.c_int(0)
    _check(lib().pw_commit(ctx, C.byref(n)), ctx)
    return n.value


def pw_sync_io(ctx):
    _check(lib().pw_sync_io(ctx), ctx)


def pw_query(ctx, block) -> pw_block_info:
    info = pw_block_info()
    _check(lib().pw_query(ctx, block, C.byref(info)), ctx)
    return info


def pw_memory(ctx) -> pw_mem_info:
    info = pw_mem_info()
    _check(lib().pw_memory(ctx, C.byref(info)), ctx)
    return info


def pw_set_fault(ctx, kind, n):
    _check(lib().pw_set_fault(ctx, kind, n), ctx)


def pw_route_noalloc(ctx, layer, x, T, ids, w, flags=0, stream=None):
    _check(lib().pw_route_noalloc(ctx, layer, _ptr(x), T, _ptr(ids), _ptr(w), flags, _stream(stream)), ctx)


def pw_set_gemv_tokens(ctx, max_tokens):
    _check(lib().pw_set_gemv_tokens(ctx, int(max_tokens)), ctx)


def pw_set_profiling(ctx, on):
    _check(lib().pw_set_profiling(ctx, int(on)), ctx)


def pw_profile_read(ctx, layer):
    ms = np.zeros(4, dtype=np.float32)
    _check(lib().pw_profile_read(ctx, layer, _ptr(ms)), ctx)
    return ms


def pw_tc_selftest(A, B, N, K, D, err, stream=None, a_in_tmem=False):
    _check(lib().pw_tc_selftest(_ptr(A), _ptr(B), N, K, 1 if a_in_tmem else 0, _ptr(D), _ptr(err), _stream(stream)))


def pw_unpack_indices(ctx, block, b, N, K):
    out = np.zeros((N, K), dtype=np.uint8)
    _check(lib().pw_unpack_indices(ctx, block, b, _ptr(out)), ctx)
    return out


def pw_dequant(ctx, block, b, N, K):
    out = np.zeros((N, K), dtype=np.uint16)
    _check(lib().pw_dequant(ctx, block, b, _ptr(out)), ctx)
    return out


def pw_pack_planes_host(idx: np.ndarray, bmax: int) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.uint8)
    N, K = idx.shape
    W = (K + 127) // 128 * 4
    out = np.zeros((bmax, N, W), dtype=np.uint32)
    _check(lib().pw_pack_planes_host(_ptr(idx), N, K, bmax, _ptr(out)))
    return out


def pw_tile_planes_host(planes: np.ndarray, K: int, u: int) -> np.ndarray:
    planes = np.ascontiguousarray(planes, dtype=np.uint32)
    nplanes, N, W = planes.shape
    out = np.zeros_like(planes)
    _check(lib().pw_tile_planes_host(_ptr(planes), N, K, nplanes, u, _ptr(out)))
    return out


def pw_untile_planes_host(tiled: np.ndarray, K: int, u: int) -> np.ndarray:
    tiled = np.ascontiguousarray(tiled, dtype=np.uint32)
    nplanes, N, W = tiled.shape
    out = np.zeros_like(tiled)
    _check(lib().pw_untile_planes_host(_ptr(tiled), N, K, nplanes, u, _ptr(out)))
    return out


def _plan_result(plan, entries):
    return dict(kind=plan.kind, stage=plan.stage, D=plan.D, total=plan.total,
                entries=[(entries[i].block, entries[i].from_bits, entries[i].to_bits, entries[i].delta)
                         for i in range(plan.n)])


def _offline_struct(off, keep):
    def arr(v, dt):
        a = np.ascontiguousarray(v, dtype=dt)
        keep.append(a)
        return a.ctypes.data
    return pw_offline(n_bits=int(np.asarray(off["s"]).shape[1]), s=arr(off["s"], np.float64),
                      head_w=arr(off["head_w"], np.float64), head_a=arr(off["head_a"], np.float64),
                      head_c=arr(off["head_c"], np.float64), alpha=float(off["alpha"]),
                      rho_min=float(off["rho_min"]), rho_max=float(off["rho_max"]), eps=float(off["eps"]),
                      n_buckets=len(off["mu"]), mu=arr(off["mu"], np.float64),
                      floors=arr(off["floors"], np.int32), n_stages=int(off["n_stages"]))


def pw_plan_host(bits, q, q_init, utype, layer, expert, M, L, E, obs: dict, off: dict, capacity=None):
    keep = []

    def arr(v, dt):
        a = np.ascontiguousarray(v, dtype=dt)
        keep.append(a)
        return a.ctypes.data
    n = len(q)
    prob = pw_plan_problem(n_blocks=n, n_bits=len(bits), L=L, E=E, bits=arr(bits, np.int32), q=arr(q, np.int32),
                           q_init=arr(q_init, np.int32), utype=arr(utype, np.int32), layer=arr(layer, np.int32),
                           expert=arr(expert, np.int32), M=arr(M, np.float64))
    o = pw_obs(T_blk=int(obs["T_blk"]), F_blk=int(obs["F_blk"]), B_KV=float(obs["B_KV"]), R=int(obs.get("R", 0)),
               mass=arr(obs["mass"], np.float64),
               phi=arr(obs["phi"], np.float64) if obs.get("phi") is not None else None,
               rho_hat=arr(obs["rho_hat"], np.float64) if obs.get("rho_hat") is not None else None)
    f = _offline_struct(off, keep)
    cap = capacity if capacity is not None else max(n, 1)
    entries = (pw_plan_entry * cap)()
    plan = pw_plan(entries=C.cast(entries, C.POINTER(pw_plan_entry)), capacity=cap)
    _check(lib().pw_plan_host(C.byref(prob), C.byref(o), C.byref(f), C.byref(plan)))
    return _plan_result(plan, entries)


def pw_plan_step(ctx, n_blocks, obs: dict, off: dict):
    keep = []

    def arr(v, dt):
        a = np.ascontiguousarray(v, dtype=dt)
        keep.append(a)
        return a.ctypes.data
    o = pw_obs(T_blk=int(obs["T_blk"]), F_blk=int(obs["F_blk"]), B_KV=float(obs["B_KV"]), R=int(obs.get("R", 0)),
               mass=arr(obs["mass"], np.float64) if obs.get("mass") is not None else None,
               phi=arr(obs["phi"], np.float64) if obs.get("phi") is not None else None,
               rho_hat=arr(obs["rho_hat"], np.float64) if obs.get("rho_hat") is not None else None)
    f = _offline_struct(off, keep)
    entries = (pw_plan_entry * n_blocks)()
    plan = pw_plan(entries=C.cast(entries, C.POINTER(pw_plan_entry)), capacity=n_blocks)
    _check(lib().pw_plan_step(ctx, C.byref(o), C.byref(f), C.byref(plan)), ctx)
    return _plan_result(plan, entries)


def pw_merge_requests(requests, kv_blocks, L, E, n_blocks, n_bits):
    """requests: dicts with mass [L][E], rho_hat [n_blocks][n_bits-1], conf [2][n_bits-1],
    rho_min, rho_max; kv_blocks: one weight per request.  Returns the merged table as a dict."""
    keep = []

    def arr(v):
        a = np.ascontiguousarray(v, dtype=np.float64)
        keep.append(a)
        return a.ctypes.data
    reqs = (pw_request_signals * len(requests))()
    for r, (q, kv) in enumerate(zip(requests, kv_blocks)):
        reqs[r] = pw_request_signals(mass=arr(q["mass"]), rho_hat=arr(q["rho_hat"]), conf=arr(q["conf"]),
                                     rho_min=float(q["rho_min"]), rho_max=float(q["rho_max"]), kv_blocks=float(kv))
    mass = np.zeros((L, E))
    rho = np.zeros((n_blocks, n_bits - 1))
    conf = np.zeros((2, n_bits - 1))
    lo, hi = C.c_double(), C.c_double()
    _check(lib().pw_merge_requests(reqs, len(requests), L, E, n_blocks, n_bits, _ptr(mass), _ptr(rho), _ptr(conf),
                                   C.byref(lo), C.byref(hi)))
    return dict(mass=mass, rho_hat=rho, conf=conf, rho_min=lo.value, rho_max=hi.value)


# ---------------------------------------------------------------- KV-block allocator
def pw_kv_create(budget_bytes, block_bytes):
    """A KV-block allocator over `budget_bytes` shared with the weight pages (handle)."""
    kv = C.c_void_p()
    _check(lib().pw_kv_create(int(budget_bytes), int(block_bytes), C.byref(kv)))
    return kv


def pw_kv_destroy(kv):
    lib().pw_kv_destroy(kv)


def pw_kv_set_weight_bytes(kv, weight_bytes):
    _check(lib().pw_kv_set_weight_bytes(kv, int(weight_bytes)))


def pw_kv_attach(kv, ctx):
    _check(lib().pw_kv_attach(kv, ctx))


def pw_kv_announce(kv, request, n_blocks):
    _check(lib().pw_kv_announce(kv, int(request), int(n_blocks)))


def pw_kv_grow(kv, request, n_blocks) -> np.ndarray:
    """Grow a request; returns the granted block ids (int32).  PwError(PW_ERR_OOM) when the
    free blocks do not suffice."""
    ids = np.zeros(max(int(n_blocks), 1), dtype=np.int32)
    _check(lib().pw_kv_grow(kv, int(request), int(n_blocks), ids.ctypes.data))
    return ids[:int(n_blocks)]


def pw_kv_release(kv, request) -> int:
    n = C.c_int64()
    _check(lib().pw_kv_release(kv, int(request), C.byref(n)))
    return n.value


def pw_kv_request(kv, request):
    """(blocks held, blocks announced) of a request."""
    held, ann = C.c_int64(), C.c_int64()
    _check(lib().pw_kv_request(kv, int(request), C.byref(held), C.byref(ann)))
    return held.value, ann.value


def pw_kv_blocks(kv, request) -> np.ndarray:
    n = C.c_int64()
    _check(lib().pw_kv_blocks(kv, int(request), None, 0, C.byref(n)))
    ids = np.zeros(max(n.value, 1), dtype=np.int32)
    _check(lib().pw_kv_blocks(kv, int(request), ids.ctypes.data, n.value, C.byref(n)))
    return ids[:n.value]


def pw_kv_get_stats(kv) -> dict:
    st = pw_kv_stats()
    _check(lib().pw_kv_get_stats(kv, C.byref(st)))
    return {name: getattr(st, name) for name, _ in pw_kv_stats._fields_}
