"""KDA oracle: fp64 CPU reference of the Kimi Delta Attention recurrence.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import this package.  The
CUDA product path never imports, links or calls it, and it imports nothing
from the product package.

Three forms live here, each written independently of the others:

* ``prefill`` -- the C library ``kda_oracle.c``: the page's three-line update
  (forget gating, predict, memory updating) and o_t = S_t q_t, one token at a
  time in fp64 ("Kimi (AI)", section "Kimi Delta Attention (KDA)").
* ``backward`` -- the same C library, reverse mode of that update: the
  gradients of sum(dO * o) + sum(dS_T * S_T) with respect to q, k, v, alpha,
  beta and S0, one token at a time in fp64.
* ``dense_form.run`` -- numpy, tiny sizes only: the same recurrence expanded
  into one explicit matrix product per step,
  S_t = diag(alpha_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T.

``attnres`` (numpy, fp64) is the reference of a second workload on the same
page, Attention Residuals, plain and blocked ("Kimi (AI)", section
"Attention Residuals").
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")

# Flags are part of the oracle's definition: strict IEEE fp64, no contraction.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra"]

KIND_BF16 = 0
KIND_F32 = 1

_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle with gcc if the library is missing or stale; return its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src)
            and not extra_flags):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, *extra_flags, src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) the oracle library and declare its signatures."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    lib = ctypes.CDLL(path or build())
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.kda_oracle_prefill.restype = ctypes.c_int
    lib.kda_oracle_prefill.argtypes = [vp, vp, vp, ctypes.c_int, vp, vp, vp, vp, i32, i64,
                                       i32, i32, i32, vp, vp, i32]
    lib.kda_oracle_prefill_additive.restype = ctypes.c_int
    lib.kda_oracle_prefill_additive.argtypes = lib.kda_oracle_prefill.argtypes
    lib.kda_oracle_backward.restype = ctypes.c_int
    lib.kda_oracle_backward.argtypes = [vp, vp, vp, ctypes.c_int, vp, vp, vp, vp, i32, i64,
                                        i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, i32]
    lib.kda_oracle_max_threads.restype = ctypes.c_int
    lib.kda_oracle_max_threads.argtypes = []
    if path is None:
        _lib = lib
    return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _as_qkv(x: np.ndarray):
    if x.dtype == np.uint16:
        return np.ascontiguousarray(x), KIND_BF16
    if x.dtype == np.float32:
        return np.ascontiguousarray(x), KIND_F32
    raise TypeError("q, k, v must be bf16 bit patterns (uint16) or float32, got %s" % x.dtype)


def prefill(q, k, v, alpha, beta, S0, cu_seqlens, *, nthreads: int = 0, lib=None,
            additive: bool = False):
    """Run the recurrence over a packed batch.

    q, k: [T_total, H, d_k]; v: [T_total, H, d_v] (uint16 bf16 bits or float32,
    all three the same).  alpha: [T_total, H, d_v] float32; beta: [T_total, H]
    float32; S0: [N, H, d_v, d_k] float64 or None (zeros); cu_seqlens: [N+1]
    int32.  Returns (o [T_total, H, d_v] float64, S_T [N, H, d_v, d_k] float64).
    Tokens past cu_seqlens[-1] get o = 0.  additive=True runs the additive
    update of linear attention instead of the delta rule (no predict step:
    S_t = diag(alpha_t) S_{t-1} + beta_t v_t k_t^T), the page's naive linear
    attention when alpha = beta = 1.
    """
    lib = lib or load()
    q, kind = _as_qkv(q)
    k, kind_k = _as_qkv(k)
    v, kind_v = _as_qkv(v)
    if not (kind == kind_k == kind_v):
        raise TypeError("q, k and v must share one storage type")
    T, H, d_k = q.shape
    d_v = v.shape[2]
    alpha = np.ascontiguousarray(alpha, dtype=np.float32)
    beta = np.ascontiguousarray(beta, dtype=np.float32)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    N = cu.shape[0] - 1
    if k.shape != (T, H, d_k) or v.shape != (T, H, d_v) or alpha.shape != (T, H, d_v) \
            or beta.shape != (T, H):
        raise ValueError("inconsistent shapes")
    if S0 is not None:
        S0 = np.ascontiguousarray(S0, dtype=np.float64)
        if S0.shape != (N, H, d_v, d_k):
            raise ValueError("S0 must be [N, H, d_v, d_k]")
    o = np.zeros((T, H, d_v), dtype=np.float64)
    S_T = np.zeros((N, H, d_v, d_k), dtype=np.float64)
    fn = lib.kda_oracle_prefill_additive if additive else lib.kda_oracle_prefill
    rc = fn(_ptr(q), _ptr(k), _ptr(v), kind, _ptr(alpha), _ptr(beta), _ptr(S0), _ptr(cu), N,
            T, H, d_k, d_v, _ptr(o), _ptr(S_T), int(nthreads))
    if rc != 0:
        raise ValueError("kda_oracle_prefill failed with code %d" % rc)
    return o, S_T


def backward(q, k, v, alpha, beta, S0, cu_seqlens, dO, dS_T=None, *, nthreads: int = 0,
             lib=None):
    """Gradients of L = sum(dO * o) + sum(dS_T * S_T) for the batch ``prefill`` runs.

    Inputs as for ``prefill``; dO: [T_total, H, d_v] and dS_T: [N, H, d_v, d_k]
    or None (zeros), any float type, widened to fp64.  Returns a dict of fp64
    arrays: dq, dk [T_total, H, d_k]; dv, dalpha [T_total, H, d_v];
    dbeta [T_total, H]; dS0 [N, H, d_v, d_k].  Reverse mode of the page's
    three-line update, one token at a time ("Kimi (AI)", section "Kimi Delta
    Attention (KDA)"); see ``kda_oracle_backward`` in ``kda_oracle.c``.
    """
    lib = lib or load()
    q, kind = _as_qkv(q)
    k, kind_k = _as_qkv(k)
    v, kind_v = _as_qkv(v)
    if not (kind == kind_k == kind_v):
        raise TypeError("q, k and v must share one storage type")
    T, H, d_k = q.shape
    d_v = v.shape[2]
    alpha = np.ascontiguousarray(alpha, dtype=np.float32)
    beta = np.ascontiguousarray(beta, dtype=np.float32)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    N = cu.shape[0] - 1
    if k.shape != (T, H, d_k) or v.shape != (T, H, d_v) or alpha.shape != (T, H, d_v) \
            or beta.shape != (T, H):
        raise ValueError("inconsistent shapes")
    dO = np.ascontiguousarray(dO, dtype=np.float64)
    if dO.shape != (T, H, d_v):
        raise ValueError("dO must be [T, H, d_v]")
    if S0 is not None:
        S0 = np.ascontiguousarray(S0, dtype=np.float64)
        if S0.shape != (N, H, d_v, d_k):
            raise ValueError("S0 must be [N, H, d_v, d_k]")
    if dS_T is not None:
        dS_T = np.ascontiguousarray(dS_T, dtype=np.float64)
        if dS_T.shape != (N, H, d_v, d_k):
            raise ValueError("dS_T must be [N, H, d_v, d_k]")
    out = {
        "dq": np.zeros((T, H, d_k)), "dk": np.zeros((T, H, d_k)),
        "dv": np.zeros((T, H, d_v)), "dalpha": np.zeros((T, H, d_v)),
        "dbeta": np.zeros((T, H)), "dS0": np.zeros((N, H, d_v, d_k)),
    }
    rc = lib.kda_oracle_backward(_ptr(q), _ptr(k), _ptr(v), kind, _ptr(alpha), _ptr(beta),
                                 _ptr(S0), _ptr(cu), N, T, H, d_k, d_v, _ptr(dO), _ptr(dS_T),
                                 _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
                                 _ptr(out["dalpha"]), _ptr(out["dbeta"]), _ptr(out["dS0"]),
                                 int(nthreads))
    if rc != 0:
        raise ValueError("kda_oracle_backward failed with code %d" % rc)
    return out


def decode_step(q, k, v, alpha, beta, S, additive: bool = False, *, lib=None):
    """One recurrent step for B independent sequences.

    q, k: [B, H, d_k]; v, alpha: [B, H, d_v]; beta: [B, H]; S: [B, H, d_v, d_k]
    (any float type, widened to fp64).  Returns (o [B, H, d_v], S_new) in fp64.
    A decode step is the recurrence over sequences of length one.
    """
    B = q.shape[0]
    cu = np.arange(B + 1, dtype=np.int32)
    return prefill(q, k, v, alpha, beta, np.asarray(S, dtype=np.float64), cu, lib=lib,
                   additive=additive)


def max_threads(lib=None) -> int:
    return int((lib or load()).kda_oracle_max_threads())


def bf16_bits_to_f64(x: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
