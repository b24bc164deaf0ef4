"""ctypes wrapper around the plain-C CPU oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``.  The GPU library and its Python
binding never import this package.  The oracle shares no code with the GPU
path; see ``moe_oracle.c`` for the citations and the parity status of every
function.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

DT_F32, DT_BF16 = 0, 1
SLOT_KEPT, SLOT_REROUTED, SLOT_DROPPED = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, no contraction of a*b+c;
    OpenMP over independent tokens and experts)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
               _SRC, "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            c_i, c_f, c_p = ctypes.c_int, ctypes.c_float, ctypes.c_void_p
            L.orc_set_threads.restype = None
            L.orc_set_threads.argtypes = [c_i]
            L.orc_get_threads.restype = c_i
            L.orc_get_threads.argtypes = []
            L.orc_exp_spec.restype = c_f
            L.orc_exp_spec.argtypes = [c_f]
            L.orc_exp_spec_array.restype = None
            L.orc_exp_spec_array.argtypes = [c_p, c_p, ctypes.c_long]
            L.orc_exp_constants.restype = None
            L.orc_exp_constants.argtypes = [c_p]
            L.orc_router.argtypes = [c_p, c_i, c_p, c_i, c_i, c_i, c_p]
            L.orc_route.argtypes = [c_p, c_i, c_i, c_i, c_i, c_p, c_p]
            L.orc_sere.argtypes = [c_p, c_p, c_i, c_i, c_i, c_i, c_i, c_f, c_p, c_p, c_p, c_p]
            L.orc_fixed_weight.restype = ctypes.c_int64
            L.orc_fixed_weight.argtypes = [c_f]
            L.orc_capacity_value.restype = ctypes.c_int64
            L.orc_capacity_value.argtypes = [ctypes.c_int64, c_i, c_f, c_i]
            L.orc_capacity.argtypes = [c_p, c_p, c_i, c_i, c_i, c_i, c_i, c_p, c_f, c_p, c_p, c_p, c_p, c_p, c_p,
                                       c_f]
            L.orc_capacity_expert.restype = ctypes.c_int64
            L.orc_capacity_expert.argtypes = [ctypes.c_int64, c_i, c_f, c_i, c_i, c_f]
            L.orc_permute.argtypes = [c_p, c_p, c_i, c_i, c_i, c_i, c_p, c_p, c_p, c_p, c_p]
            L.orc_ffn_combine.argtypes = [c_p, c_i, c_p, c_p, c_p, c_i, c_i, c_i, c_i, c_i, c_p, c_p, c_i, c_i,
                                          c_p, c_i, c_p]
            c_d = ctypes.c_double
            L.orc_token_weights.argtypes = [c_p, c_i, c_i, c_i, c_p, c_d, c_d, c_p, c_p, c_p]
            L.orc_similarity.argtypes = [c_p, c_i, c_i, c_i, c_p, c_p, c_p, c_i, c_i, c_i, c_p]
            _lib = L
    return _lib


def set_threads(n: int) -> int:
    """Host threads for the oracle's loops over independent tokens or experts
    (n <= 0: every host core).  Results do not depend on it.  Returns the
    count now in effect."""
    lib().orc_set_threads(int(n))
    return int(lib().orc_get_threads())


def threads() -> int:
    return int(lib().orc_get_threads())


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError("oracle %s failed with code %d" % (what, rc))


def exp_spec(d) -> np.ndarray:
    d = np.ascontiguousarray(d, dtype=np.float32)
    out = np.zeros_like(d)
    lib().orc_exp_spec_array(_p(d), _p(out), d.size)
    return out


def exp_constants() -> np.ndarray:
    out = np.zeros(11, dtype=np.float32)
    lib().orc_exp_constants(_p(out))
    return out


def router(x: np.ndarray, w_r: np.ndarray, x_dtype: int = DT_F32) -> np.ndarray:
    """Router logits [T][N] (fp32) from x [T][H] (fp32 values or bf16 bits) and w_r [N][H]."""
    x = np.ascontiguousarray(x)
    w_r = np.ascontiguousarray(w_r, dtype=np.float32)
    T, H = x.shape
    N = w_r.shape[0]
    out = np.zeros((T, N), dtype=np.float32)
    _check(lib().orc_router(_p(x), x_dtype, _p(w_r), T, H, N, _p(out)), "router")
    return out


def route(logits: np.ndarray, R: int, renorm_k: int = 0):
    """Softmax gates and the top-R ranking: ids [T][R] int32, gates [T][R] fp32."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, N = logits.shape
    ids = np.zeros((T, R), dtype=np.int32)
    gates = np.zeros((T, R), dtype=np.float32)
    _check(lib().orc_route(_p(logits), T, N, R, renorm_k, _p(ids), _p(gates)), "route")
    return ids, gates


def sere(ids: np.ndarray, gates: np.ndarray, N: int, k: int, k_primary: int, rho: float,
         sim: np.ndarray, protect=None):
    """SERE reroute on copies of ids/gates (first k columns used).
    Returns (ids, gates, bitmap of P, stats[8])."""
    ids = np.array(ids, dtype=np.int32, order="C", copy=True)
    gates = np.array(gates, dtype=np.float32, order="C", copy=True)
    T, ld = ids.shape
    sim = np.ascontiguousarray(sim, dtype=np.float32)
    prot = None if protect is None else np.ascontiguousarray(protect, dtype=np.uint8)
    bitmap = np.zeros((N + 31) // 32, dtype=np.uint32)
    stats = np.zeros(8, dtype=np.int32)
    _check(lib().orc_sere(_p(ids), _p(gates), ld, T, N, k, k_primary, float(rho), _p(sim), _p(prot),
                          _p(bitmap), _p(stats)), "sere")
    return ids, gates, bitmap, stats


def fixed_weight(w: float) -> int:
    return int(lib().orc_fixed_weight(float(w)))


def capacity_value(S: int, k: int, gamma: float, N: int) -> int:
    return int(lib().orc_capacity_value(int(S), k, float(gamma), N))


def capacity(ids: np.ndarray, gates: np.ndarray, N: int, k: int, R: int, token_w, gamma: float,
             bias=None, r_v: float = 0.5):
    """Capacity dispatch.  Returns (out_ids [T][k], out_gates [T][k], status [T][k], load [N], C) with C the
    static capacity.  With `bias` ([N] int8 modality bias m_j) each expert's capacity is
    capacity_expert(S, k, gamma, N, m_j, r_v) instead."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    gates = np.ascontiguousarray(gates, dtype=np.float32)
    T, ld = ids.shape
    tw = None if token_w is None else np.ascontiguousarray(token_w, dtype=np.float32)
    bs = None if bias is None else np.ascontiguousarray(bias, dtype=np.int8)
    out_ids = np.zeros((T, k), dtype=np.int32)
    out_gates = np.zeros((T, k), dtype=np.float32)
    status = np.zeros((T, k), dtype=np.uint8)
    load = np.zeros(N, dtype=np.int64)
    cap = np.zeros(1, dtype=np.int64)
    _check(lib().orc_capacity(_p(ids), _p(gates), ld, T, N, k, R, _p(tw), float(gamma), _p(out_ids),
                              _p(out_gates), _p(status), _p(load), _p(cap), _p(bs), float(r_v)), "capacity")
    return out_ids, out_gates, status, load, int(cap[0])


def capacity_expert(S: int, k: int, gamma: float, N: int, m: int, r_v: float) -> int:
    """Per-expert capacity (a reading of the truncated [MACS] 3.3):
    floor(c * (1 + m (r_v - 1/2))) with c the unfloored static capacity."""
    return int(lib().orc_capacity_expert(int(S), k, float(gamma), N, int(m), float(r_v)))


def permute(ids: np.ndarray, gates: np.ndarray, N: int, k: int):
    """Rows in (expert asc, token asc) order.  Returns dict of counts, offsets,
    row_token, row_gate, active (active[0] = count)."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    gates = np.ascontiguousarray(gates, dtype=np.float32)
    T, ld = ids.shape
    M = T * k
    counts = np.zeros(N, dtype=np.int32)
    offsets = np.zeros(N + 1, dtype=np.int32)
    row_token = np.full(max(M, 1), -1, dtype=np.int32)
    row_gate = np.zeros(max(M, 1), dtype=np.float32)
    active = np.zeros(N + 1, dtype=np.int32)
    _check(lib().orc_permute(_p(ids), _p(gates), ld, T, N, k, _p(counts), _p(offsets), _p(row_token),
                             _p(row_gate), _p(active)), "permute")
    m = int(offsets[N])
    return dict(counts=counts, offsets=offsets, row_token=row_token[:m], row_gate=row_gate[:m], active=active)


def ffn_combine(x, w_gate, w_up, w_down, ids, gates, k: int, tokens=None, x_dtype: int = DT_F32,
                w_dtype: int = DT_F32) -> np.ndarray:
    """y [len(tokens)][H] in float64 for the listed tokens (all tokens by default)."""
    x = np.ascontiguousarray(x)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    gates = np.ascontiguousarray(gates, dtype=np.float32)
    T, H = x.shape
    N, I = w_gate.shape[0], w_gate.shape[1]
    ld = ids.shape[1]
    tok = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    y = np.zeros((len(tok), H), dtype=np.float64)
    _check(lib().orc_ffn_combine(_p(x), x_dtype, _p(w_gate), _p(w_up), _p(w_down), w_dtype, T, H, I, N,
                                 _p(ids), _p(gates), ld, k, _p(tok), len(tok), _p(y)), "ffn_combine")
    return y


def token_weights(x: np.ndarray, is_visual: np.ndarray, delta: float = 1.0, eps: float = 1e-6,
                  x_dtype: int = DT_F32):
    """[MACS] Eqs. (4)-(5), (7): per-token entropy of Softmax(x_t), the
    entropy weights w and the effective visual ratio R_v (float64)."""
    x = np.ascontiguousarray(x)
    T, H = x.shape
    vis = np.ascontiguousarray(is_visual, dtype=np.uint8)
    ent = np.zeros(max(T, 1), dtype=np.float64)
    w = np.zeros(max(T, 1), dtype=np.float64)
    rv = np.zeros(1, dtype=np.float64)
    _check(lib().orc_token_weights(_p(x), x_dtype, T, H, _p(vis), float(delta), float(eps), _p(ent), _p(w),
                                   _p(rv)), "token_weights")
    return ent[:T], w[:T], float(rv[0])


def similarity(x: np.ndarray, w_gate, w_up, w_down, x_dtype: int = DT_F32, w_dtype: int = DT_F32) -> np.ndarray:
    """[SERE] 4.2: Frobenius similarity of the experts' outputs on the
    calibration tokens x [n][H]; [N][N] float64."""
    x = np.ascontiguousarray(x)
    n, H = x.shape
    N, I = w_gate.shape[0], w_gate.shape[1]
    out = np.zeros((N, N), dtype=np.float64)
    _check(lib().orc_similarity(_p(x), x_dtype, n, H, _p(np.ascontiguousarray(w_gate)), _p(np.ascontiguousarray(w_up)),
                                _p(np.ascontiguousarray(w_down)), w_dtype, I, N, _p(out)), "similarity")
    return out


def layer(L, sere_on: bool, capacity_on: bool = False, tokens=None, renorm_k: int = 0, logits=None):
    """The whole layer on the CPU for a synthetic ``Layer``: router -> top-R ->
    (SERE) -> (capacity) -> permute -> FFN + combine.  Returns a dict of every
    intermediate."""
    xd = DT_BF16 if L.dtype == "bf16" else DT_F32
    wd = DT_BF16 if L.dtype == "bf16" else DT_F32
    xin = L.x_bf16 if L.dtype == "bf16" else L.x
    out = {}
    if logits is None:
        logits = router(xin, L.w_r, xd)
    out["logits"] = logits
    R = L.R if capacity_on else L.k
    ids, gates = route(logits, R, renorm_k)
    out["ids_ranked"], out["gates_ranked"] = ids, gates
    if sere_on:
        ids_k, gates_k, bitmap, stats = sere(ids[:, :L.k], gates[:, :L.k], L.N, L.k, L.k_primary, L.rho,
                                             L.sim, L.protect)
        out["bitmap"], out["stats"] = bitmap, stats
    else:
        ids_k, gates_k = ids[:, :L.k].copy(), gates[:, :L.k].copy()
    if capacity_on:
        ids_k, gates_k, status, load, cap = capacity(ids, gates, L.N, L.k, R, L.token_w, L.gamma)
        out["status"], out["load"], out["cap"] = status, load, cap
    out["ids"], out["gates"] = ids_k, gates_k
    out["perm"] = permute(ids_k, gates_k, L.N, L.k)
    if L.w_gate is not None:
        out["y"] = ffn_combine(xin, L.w_gate, L.w_up, L.w_down, ids_k, gates_k, L.k, tokens, xd, wd)
        out["y_tokens"] = np.arange(L.T) if tokens is None else np.asarray(tokens)
    return out
