"""CPU oracle of the ZeRO optimizer step (test infrastructure).

Only the test-suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg import this package. The GPU product path never does, and the two share no
code. The arithmetic lives in ``zero_oracle.c`` (plain C, no FMA contraction); this module
only compiles it with gcc and marshals numpy arrays through ctypes.

The oracle keeps M genuinely separate rank structures (one shard of fp32 master / m / v per
owner, one bf16 replica or shard per rank), following the ZeRO-1/2/3 lifecycles of
"CS336 2026 Lecture 8" Slides 19-26 and "并行训练优化、MoE扩展与系统瓶颈" 2.2.1-2.2.6.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zero_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None

# A lane alignment of 64 elements gives every bf16 shard a 128-byte start.
DEFAULT_ALIGN = 64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build/liboracle.so (returns its path)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Hyper(ctypes.Structure):
    """AdamW + clip hyper-parameters (mirrors ``orc_hyper``)."""

    _fields_ = [
        ("lr", ctypes.c_double),
        ("beta1", ctypes.c_double),
        ("beta2", ctypes.c_double),
        ("eps", ctypes.c_double),
        ("weight_decay", ctypes.c_double),
        ("max_grad_norm", ctypes.c_double),
        ("clip", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


def hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, max_grad_norm=1.0, clip=False):
    return Hyper(lr, beta1, beta2, eps, weight_decay, max_grad_norm, 1 if clip else 0, 0)


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # ZERO_ORACLE_LIB lets the mutation test load a deliberately broken copy.
            lib = ctypes.CDLL(os.environ.get("ZERO_ORACLE_LIB") or build())
            lib.orc_plan.restype = _I64
            lib.orc_plan.argtypes = [_I32, _I64, _I64, _P, _I64, _P, _P, _P, _P, _P, _P]
            lib.orc_bf16_rne_array.restype = None
            lib.orc_bf16_rne_array.argtypes = [_P, _P, _I64]
            lib.orc_bf16_to_f32_array.restype = None
            lib.orc_bf16_to_f32_array.argtypes = [_P, _P, _I64]
            lib.orc_reduce_scatter.restype = None
            lib.orc_reduce_scatter.argtypes = [_I32, _I64, _P, _P, _P, _P, _P]
            lib.orc_global_sumsq.restype = ctypes.c_double
            lib.orc_global_sumsq.argtypes = [_I32, _I64, _P, _P, _P]
            lib.orc_sumsq_chunk.restype = ctypes.c_double
            lib.orc_sumsq_chunk.argtypes = [ctypes.c_double, _I32, _P, _I64, _I64, _I64, _P, _P]
            lib.orc_clip_scale.restype = ctypes.c_float
            lib.orc_clip_scale.argtypes = [ctypes.c_double, ctypes.c_double]
            lib.orc_adamw.restype = None
            lib.orc_adamw.argtypes = [_I64, _P, ctypes.c_float, _P, _P, _P, ctypes.POINTER(Hyper), _I64]
            lib.orc_init.restype = None
            lib.orc_init.argtypes = [_I32, _I32, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P]
            lib.orc_zero_step.restype = ctypes.c_int
            lib.orc_zero_step.argtypes = [_I32, _I32, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                          ctypes.POINTER(Hyper), _I64,
                                          ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_float)]
            lib.orc_hsdp_step.restype = ctypes.c_int
            lib.orc_hsdp_step.argtypes = [_I32, _I32, _I32, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                          ctypes.POINTER(Hyper), _I64,
                                          ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_float)]
            lib.orc_naive_dp_step_groups.restype = ctypes.c_int
            lib.orc_naive_dp_step_groups.argtypes = [_I32, _I32, _I64, _P, _P, _P, _P, _P, ctypes.POINTER(Hyper),
                                                     _I64, ctypes.POINTER(ctypes.c_double),
                                                     ctypes.POINTER(ctypes.c_float)]
            lib.orc_naive_dp_step.restype = ctypes.c_int
            lib.orc_naive_dp_step.argtypes = [_I32, _I64, _P, _P, _P, _P, _P, ctypes.POINTER(Hyper), _I64,
                                              ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_float)]
            lib.orc_lane_steps.restype = None
            lib.orc_lane_steps.argtypes = [_I32, _I64, _I32, _P, _P, _P, _P, ctypes.POINTER(Hyper), _I64,
                                           _P, _P, _P, _P, _P]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _ptr_array(arrs):
    """ctypes array of pointers to the given numpy arrays (keeps no reference; caller does)."""
    return (ctypes.c_void_p * max(len(arrs), 1))(*[a.ctypes.data for a in arrs])


# ------------------------------------------------------------------------------------------
# bf16 helpers
# ------------------------------------------------------------------------------------------
def bf16_rne(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), IEEE round-to-nearest-even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().orc_bf16_rne_array(_ptr(x), _ptr(out), x.size)
    return out


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _load().orc_bf16_to_f32_array(_ptr(h), _ptr(out), h.size)
    return out


# ------------------------------------------------------------------------------------------
# Layout
# ------------------------------------------------------------------------------------------
@dataclass
class Plan:
    """Flat bucket / shard layout computed by the oracle's own planner."""

    M: int
    A: int
    bucket_bytes: int
    numel: np.ndarray
    b_first: np.ndarray  # first tensor of each bucket (length nb + 1, last = T)
    b_off: np.ndarray    # padded start lane of each bucket
    b_n: np.ndarray      # real lanes of each bucket
    b_S: np.ndarray      # shard length of each bucket
    t_off: np.ndarray    # padded start lane of each tensor
    npad: int
    N: int = field(init=False)
    shard_len: int = field(init=False)
    nb: int = field(init=False)

    def __post_init__(self):
        self.nb = int(self.b_n.size)
        self.N = int(self.b_n.sum())
        self.shard_len = int(self.b_S.sum())

    def real_mask(self) -> np.ndarray:
        """bool[npad]: True on real lanes."""
        mask = np.zeros(self.npad, dtype=bool)
        for b in range(self.nb):
            o = int(self.b_off[b])
            mask[o:o + int(self.b_n[b])] = True
        return mask

    def unpadded_index(self) -> np.ndarray:
        """int64[npad]: unpadded position of each real lane, -1 on padding lanes."""
        u = np.full(self.npad, -1, dtype=np.int64)
        ubase = 0
        for b in range(self.nb):
            o, n = int(self.b_off[b]), int(self.b_n[b])
            u[o:o + n] = np.arange(ubase, ubase + n, dtype=np.int64)
            ubase += n
        return u

    def pad(self, x_unpadded: np.ndarray, fill=0) -> np.ndarray:
        """Scatter an unpadded vector (N values) into the padded layout."""
        out = np.full(self.npad, fill, dtype=x_unpadded.dtype)
        ubase = 0
        for b in range(self.nb):
            o, n = int(self.b_off[b]), int(self.b_n[b])
            out[o:o + n] = x_unpadded[ubase:ubase + n]
            ubase += n
        return out

    def shard_lanes(self, r: int) -> np.ndarray:
        """int64[shard_len]: padded lanes owned by rank r, in shard order."""
        parts = [np.arange(int(self.b_off[b]) + r * int(self.b_S[b]),
                           int(self.b_off[b]) + (r + 1) * int(self.b_S[b]), dtype=np.int64)
                 for b in range(self.nb)]
        return np.concatenate(parts) if parts else np.zeros(0, dtype=np.int64)


def plan(numel, M: int, bucket_bytes: int = 0, A: int = DEFAULT_ALIGN) -> Plan:
    numel = np.ascontiguousarray(numel, dtype=np.int64)
    T = int(numel.size)
    cap = max(T, 1)
    b_first = np.zeros(cap + 1, dtype=np.int64)
    b_off = np.zeros(cap, dtype=np.int64)
    b_n = np.zeros(cap, dtype=np.int64)
    b_S = np.zeros(cap, dtype=np.int64)
    t_off = np.zeros(cap, dtype=np.int64)
    nb = ctypes.c_int64(0)
    npad = _load().orc_plan(M, A, bucket_bytes, _ptr(numel), T, _ptr(b_first), _ptr(b_off), _ptr(b_n),
                            _ptr(b_S), _ptr(t_off), ctypes.cast(ctypes.pointer(nb), ctypes.c_void_p))
    k = nb.value
    return Plan(M, A, bucket_bytes, numel, b_first[:k + 1].copy(), b_off[:k].copy(), b_n[:k].copy(),
                b_S[:k].copy(), t_off[:T].copy(), int(npad))


# ------------------------------------------------------------------------------------------
# Collectives and the norm
# ------------------------------------------------------------------------------------------
def reduce_scatter(p: Plan, grads) -> list:
    """Owner shards of the averaged gradient: list of M float32 arrays (shard_len each)."""
    g = [np.ascontiguousarray(x, dtype=np.uint16) for x in grads]
    assert len(g) == p.M and all(x.size == p.npad for x in g)
    out = [np.empty(p.shard_len, dtype=np.float32) for _ in range(p.M)]
    gp, op = _ptr_array(g), _ptr_array(out)
    _load().orc_reduce_scatter(p.M, p.nb, _ptr(p.b_off), _ptr(p.b_n), _ptr(p.b_S), gp, op)
    return out


def global_sumsq(p: Plan, ghat_shards) -> float:
    gs = [np.ascontiguousarray(x, dtype=np.float32) for x in ghat_shards]
    return float(_load().orc_global_sumsq(p.M, p.nb, _ptr(p.b_n), _ptr(p.b_S), _ptr_array(gs)))


def sumsq_chunk(acc: float, p: Plan, grads_chunk, o0: int) -> float:
    """Continue the fp64 sum of squared averaged gradients over lanes [o0, o0+len)."""
    g = [np.ascontiguousarray(x, dtype=np.uint16) for x in grads_chunk]
    n = int(g[0].size)
    assert len(g) == p.M and all(x.size == n for x in g)
    return float(_load().orc_sumsq_chunk(acc, p.M, _ptr_array(g), o0, n, p.nb, _ptr(p.b_off), _ptr(p.b_n)))


def clip_scale(norm: float, max_grad_norm: float) -> float:
    return float(_load().orc_clip_scale(norm, max_grad_norm))


def adamw(ghat: np.ndarray, s: float, p: np.ndarray, m: np.ndarray, v: np.ndarray, h: Hyper, t: int):
    """In-place AdamW over flat fp32 arrays."""
    for a in (ghat, p, m, v):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    _load().orc_adamw(p.size, _ptr(ghat), s, _ptr(p), _ptr(m), _ptr(v), ctypes.byref(h), t)


# ------------------------------------------------------------------------------------------
# Full ZeRO step over M rank structures
# ------------------------------------------------------------------------------------------
@dataclass
class RankState:
    """Per-rank structures of the emulated job."""

    stage: int
    master: list
    mom: list
    var: list
    ghat: list
    param: list  # stage 1/2: full bf16 replicas (N); stage 3: bf16 shards (shard_len)
    t: int = 0   # steps taken
    groups: int = 1  # hybrid sharding: G groups of p.M owners each (structures grp * p.M + k)


def init_state(p: Plan, stage: int, master_init: np.ndarray, m_init=None, v_init=None, t: int = 0,
               groups: int = 1) -> RankState:
    """Rank structures from unpadded state (m, v default to zeros; t = steps already taken).
    With groups > 1 (hybrid sharding) p is planned for the K owners of one group and every
    group gets its own copy of the K structures."""
    assert stage in (1, 2, 3)
    if groups > 1:
        one = init_state(p, stage, master_init, m_init, v_init, t)
        copies = [init_state(p, stage, master_init, m_init, v_init, t) for _ in range(groups - 1)]
        for c in copies:
            for f in ("master", "mom", "var", "ghat", "param"):
                getattr(one, f).extend(getattr(c, f))
        one.groups = groups
        return one
    mi = np.ascontiguousarray(master_init, dtype=np.float32)
    assert mi.size == p.N
    mm = None if m_init is None else np.ascontiguousarray(m_init, dtype=np.float32)
    vv = None if v_init is None else np.ascontiguousarray(v_init, dtype=np.float32)
    assert (mm is None or mm.size == p.N) and (vv is None or vv.size == p.N)
    L = max(p.shard_len, 1)
    master = [np.empty(L, dtype=np.float32) for _ in range(p.M)]
    mom = [np.empty(L, dtype=np.float32) for _ in range(p.M)]
    var = [np.empty(L, dtype=np.float32) for _ in range(p.M)]
    ghat = [np.zeros(L, dtype=np.float32) for _ in range(p.M)]
    plen = L if stage == 3 else max(p.N, 1)
    param = [np.empty(plen, dtype=np.uint16) for _ in range(p.M)]
    _load().orc_init(p.M, stage, p.nb, _ptr(p.b_n), _ptr(p.b_S), _ptr(mi), _ptr(mm) if mm is not None else None,
                     _ptr(vv) if vv is not None else None, _ptr_array(master), _ptr_array(mom), _ptr_array(var),
                     _ptr_array(param))
    return RankState(stage, master, mom, var, ghat, param, t)


def zero_step(p: Plan, st: RankState, grads, h: Hyper):
    """One ZeRO step (hybrid-sharded when st.groups > 1, with groups * p.M rank gradients);
    returns (full bf16 params [N] as uint16, norm, scale, rc)."""
    g = [np.ascontiguousarray(x, dtype=np.uint16) for x in grads]
    assert len(g) == p.M * st.groups and all(x.size == p.npad for x in g)
    full = np.empty(max(p.N, 1), dtype=np.uint16)
    norm, scale = ctypes.c_double(0.0), ctypes.c_float(0.0)
    st.t += 1
    args = (p.nb, _ptr(p.b_off), _ptr(p.b_n), _ptr(p.b_S), _ptr_array(g), _ptr_array(st.master),
            _ptr_array(st.mom), _ptr_array(st.var), _ptr_array(st.ghat), _ptr_array(st.param), _ptr(full),
            ctypes.byref(h), st.t, ctypes.byref(norm), ctypes.byref(scale))
    if st.groups > 1:
        rc = _load().orc_hsdp_step(st.groups, p.M, st.stage, *args)
    else:
        rc = _load().orc_zero_step(p.M, st.stage, *args)
    if rc < 0:
        raise AssertionError("oracle: gathered replicas disagree")
    return full[:p.N], norm.value, scale.value, rc


def flat_state(p: Plan, st: RankState, which: str) -> np.ndarray:
    """Owner shards of 'master' | 'mom' | 'var' | 'ghat' laid back into the padded layout."""
    arrs = getattr(st, which)
    out = np.zeros(p.npad, dtype=np.float32)
    for r in range(p.M):
        out[p.shard_lanes(r)] = arrs[r][:p.shard_len]
    return out


@dataclass
class DPState:
    master: list
    mom: list
    var: list
    param: list
    t: int = 0


def naive_dp_init(M: int, master_init: np.ndarray) -> DPState:
    mi = np.ascontiguousarray(master_init, dtype=np.float32)
    n = max(mi.size, 1)
    master = [mi.copy() if mi.size else np.zeros(1, np.float32) for _ in range(M)]
    mom = [np.zeros(n, dtype=np.float32) for _ in range(M)]
    var = [np.zeros(n, dtype=np.float32) for _ in range(M)]
    param = [bf16_rne(m) for m in master]
    return DPState(master, mom, var, param)


def naive_dp_step(st: DPState, grads_unpadded, h: Hyper, groups: int = 1):
    """One naive-DP step on full replicas (all-reduce summed group by group when groups > 1);
    returns (bf16 params, norm, scale, rc)."""
    g = [np.ascontiguousarray(x, dtype=np.uint16) for x in grads_unpadded]
    M = len(g)
    N = int(g[0].size)
    norm, scale = ctypes.c_double(0.0), ctypes.c_float(0.0)
    st.t += 1
    rc = _load().orc_naive_dp_step_groups(M, groups, N, _ptr_array(g), _ptr_array(st.master), _ptr_array(st.mom),
                                          _ptr_array(st.var), _ptr_array(st.param), ctypes.byref(h), st.t,
                                          ctypes.byref(norm), ctypes.byref(scale))
    if rc < 0:
        raise AssertionError("oracle: naive-DP replicas disagree")
    return st.param[0][:N].copy(), norm.value, scale.value, rc


def lane_steps(M: int, g: np.ndarray, real: np.ndarray, scales, apply, h: Hyper, t0: int,
               p: np.ndarray, m: np.ndarray, v: np.ndarray, want_ghat: bool = False):
    """Trajectories of L sampled lanes over K steps.

    g: uint16 [K, M, L]; real: bool [L]; scales/apply: [K]; p/m/v: float32 [L] (in/out).
    Returns (bf16 params [L], ghat [K, L] or None).
    """
    g = np.ascontiguousarray(g, dtype=np.uint16)
    K, Mg, L = g.shape
    assert Mg == M
    real8 = np.ascontiguousarray(real, dtype=np.uint8)
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    ap = np.ascontiguousarray(apply, dtype=np.uint8)
    for a in (p, m, v):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"] and a.size == L
    bf = np.empty(L, dtype=np.uint16)
    gh = np.empty((K, L), dtype=np.float32) if want_ghat else None
    _load().orc_lane_steps(M, L, K, _ptr(g), _ptr(real8), _ptr(sc), _ptr(ap), ctypes.byref(h), t0,
                           _ptr(p), _ptr(m), _ptr(v), _ptr(bf), _ptr(gh) if gh is not None else None)
    return bf, gh
