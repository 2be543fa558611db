"""fp64 CPU oracle for packed DAG attention -- TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and the CPU-baseline leg of bench.py may
import this package.  The library (packed_tree_attention_gb300) never does, and this
package imports nothing from it: the two share only the seeded input generators in
``synth``.

The C++ model lives in ``oracle.cpp`` (built by :func:`build` with g++ -fopenmp);
this file is a thin ctypes wrapper around it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

OK, EINVAL, ENOMEM, ESTATE = 0, 1, 2, 3


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "oracle.cpp")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fopenmp", "-shared", "-fPIC",
                               src, "-o", tmp])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        P = ctypes.c_void_p
        I = ctypes.c_int
        IP = ctypes.POINTER(ctypes.c_int)
        DP = ctypes.POINTER(ctypes.c_double)
        UP = ctypes.POINTER(ctypes.c_ubyte)
        L.orc_new.restype = P
        L.orc_new.argtypes = [I, I, I, I]
        L.orc_delete.argtypes = [P]
        L.orc_root.argtypes = [P, IP]
        L.orc_append.argtypes = [P, I, I, DP, DP, IP]
        L.orc_fork.argtypes = [P, I, I, IP]
        L.orc_mount.argtypes = [P, I, I, I, I, IP]
        L.orc_rewind.argtypes = [P, I, I, IP]
        L.orc_done.argtypes = [P, I]
        L.orc_release.argtypes = [P, I]
        L.orc_unpin.argtypes = [P, I]
        L.orc_num_segments.argtypes = [P]
        L.orc_free_pages.argtypes = [P]
        L.orc_num_mounts.argtypes = [P]
        L.orc_seg_info.argtypes = [P, I, IP]
        L.orc_seg_pos.argtypes = [P, I, IP]
        L.orc_seg_pages.argtypes = [P, I, IP]
        L.orc_mount_info.argtypes = [P, I, IP]
        L.orc_pack.restype = P
        L.orc_pack.argtypes = [P, IP, I, I, I, IP]
        L.orc_plan_total_pairs.restype = ctypes.c_longlong
        L.orc_plan_total_pairs.argtypes = [P]
        L.orc_plan_delete.argtypes = [P]
        L.orc_plan_size.restype = ctypes.c_longlong
        L.orc_plan_size.argtypes = [P, I]
        L.orc_plan_arrays.argtypes = [P] + [IP] * 10
        L.orc_fwd.argtypes = [P, I, DP, ctypes.c_double, IP, I, DP, DP, I]
        L.orc_bwd.argtypes = [P, I, DP, DP, ctypes.c_double, UP, UP, DP, DP, DP, I, I]
        L.orc_decode.argtypes = [P, IP, I, I, DP, ctypes.c_double, DP, DP]
        L.orc_row_context.argtypes = [P, I, IP, IP, I]
        L.orc_token_owner.argtypes = [P, IP, IP]
        L.orc_num_tokens.argtypes = [P]
        L.orc_set_kv.argtypes = [P, I, IP, DP, DP]
        L.orc_rope.argtypes = [DP, I, I, I, IP, ctypes.c_double, I]
        _lib = L
    return _lib


def _ip(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int)) if a is not None else None


def _dp(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double)) if a is not None else None


def _up(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)) if a is not None else None


class OracleError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: oracle status {code}")
        self.code = code


class Oracle:
    """Episode state: segments, mounts, page allocator and the K/V of every token."""

    def __init__(self, page_size: int, num_pages: int, n_kv_heads: int, head_dim: int):
        self._L = _load()
        self.h = self._L.orc_new(page_size, num_pages, n_kv_heads, head_dim)
        self.P, self.num_pages, self.Hkv, self.d = page_size, num_pages, n_kv_heads, head_dim

    def __del__(self):
        if getattr(self, "h", None):
            self._L.orc_delete(self.h)
            self.h = None

    def _chk(self, st, what):
        if st != OK:
            raise OracleError(st, what)

    # -- primitives: each returns the status; raise=True raises on failure --
    def root(self):
        out = ctypes.c_int()
        self._chk(self._L.orc_root(self.h, ctypes.byref(out)), "root")
        return out.value

    def append(self, c, n, k=None, v=None, check=True):
        pos = np.zeros(max(n, 1), dtype=np.int32)
        kk = None if k is None else np.ascontiguousarray(k, dtype=np.float64)
        vv = None if v is None else np.ascontiguousarray(v, dtype=np.float64)
        st = self._L.orc_append(self.h, c, n, _dp(kk), _dp(vv), _ip(pos))
        if check:
            self._chk(st, "append")
            return pos[:n]
        return st

    def fork(self, c, n, check=True):
        out = np.zeros(max(n, 1), dtype=np.int32)
        st = self._L.orc_fork(self.h, c, n, _ip(out))
        if check:
            self._chk(st, "fork")
            return out[:n].tolist()
        return st

    def mount(self, r, p, a, b, check=True):
        out = ctypes.c_int()
        st = self._L.orc_mount(self.h, r, p, a, b, ctypes.byref(out))
        if check:
            self._chk(st, "mount")
            return out.value
        return st

    def rewind(self, c, k, check=True):
        out = ctypes.c_int()
        st = self._L.orc_rewind(self.h, c, k, ctypes.byref(out))
        if check:
            self._chk(st, "rewind")
            return out.value
        return st

    def done(self, c, check=True):
        st = self._L.orc_done(self.h, c)
        if check:
            self._chk(st, "done")
        return st

    def release(self, c, check=True):
        st = self._L.orc_release(self.h, c)
        if check:
            self._chk(st, "release")
        return st

    def unpin(self, c, check=True):
        st = self._L.orc_unpin(self.h, c)
        if check:
            self._chk(st, "unpin")
        return st

    # -- replay of a synth.Episode op log with its K/V rows (append order) --
    def replay(self, ep, K=None, V=None):
        """Returns every appended token's position, in append order."""
        t = 0
        positions = []
        for op in ep.ops:
            kind = op[0]
            if kind == "root":
                self.root()
            elif kind == "append":
                _, c, n = op
                k = None if K is None else K[t:t + n]
                v = None if V is None else V[t:t + n]
                positions.extend(self.append(c, n, k, v).tolist())
                t += n
            elif kind == "fork":
                self.fork(op[1], op[2])
            elif kind == "mount":
                self.mount(*op[1:])
            elif kind == "rewind":
                self.rewind(op[1], op[2])
            elif kind == "done":
                self.done(op[1])
            elif kind == "release":
                self.release(op[1])
            elif kind == "unpin":
                self.unpin(op[1])
            else:
                raise ValueError(kind)
        return np.array(positions, dtype=np.int32)

    # -- queries --
    @property
    def n_segments(self):
        return self._L.orc_num_segments(self.h)

    @property
    def n_mounts(self):
        return self._L.orc_num_mounts(self.h)

    @property
    def n_tokens(self):
        return self._L.orc_num_tokens(self.h)

    def free_pages(self):
        return self._L.orc_free_pages(self.h)

    def seg_info(self, s):
        info = np.zeros(7, dtype=np.int32)
        self._chk(self._L.orc_seg_info(self.h, s, _ip(info)), "seg_info")
        keys = ("parent", "fork", "len", "n_pages", "refcount", "p_next", "flags")
        return dict(zip(keys, info.tolist()))

    def seg_pos(self, s):
        n = self.seg_info(s)["len"]
        out = np.zeros(max(n, 1), dtype=np.int32)
        self._L.orc_seg_pos(self.h, s, _ip(out))
        return out[:n]

    def seg_pages(self, s):
        n = self.seg_info(s)["n_pages"]
        out = np.zeros(max(n, 1), dtype=np.int32)
        self._L.orc_seg_pages(self.h, s, _ip(out))
        return out[:n]

    def mount_info(self, i):
        out = np.zeros(5, dtype=np.int32)
        self._chk(self._L.orc_mount_info(self.h, i, _ip(out)), "mount_info")
        return tuple(out.tolist())

    def set_kv(self, tokens, k, v):
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        k = np.ascontiguousarray(k, dtype=np.float64)
        v = np.ascontiguousarray(v, dtype=np.float64)
        self._chk(self._L.orc_set_kv(self.h, len(t), _ip(t), _dp(k), _dp(v)), "set_kv")

    def token_owner(self):
        n = self.n_tokens
        seg = np.zeros(max(n, 1), dtype=np.int32)
        idx = np.zeros(max(n, 1), dtype=np.int32)
        self._L.orc_token_owner(self.h, _ip(seg), _ip(idx))
        return seg[:n], idx[:n]

    def pack(self, roots, bm, tile_stride=1):
        """Packs the trees of `roots`; with tile_stride > 1 only every tile_stride-th
        tile gets its entries derived (the others are left empty)."""
        st = ctypes.c_int()
        r = np.ascontiguousarray(roots, dtype=np.int32)
        h = self._L.orc_pack(self.h, _ip(r), len(r), bm, tile_stride, ctypes.byref(st))
        if not h:
            raise OracleError(st.value, "pack")
        return OraclePlan(self, h, bm)

    def decode(self, cursors, q, scale):
        c = np.ascontiguousarray(cursors, dtype=np.int32)
        q = np.ascontiguousarray(q, dtype=np.float64)
        n, Hq, d = q.shape
        out = np.zeros_like(q)
        lse = np.zeros((n, Hq), dtype=np.float64)
        self._chk(self._L.orc_decode(self.h, _ip(c), n, Hq, _dp(q), scale, _dp(out), _dp(lse)), "decode")
        return out, lse


class OraclePlan:
    def __init__(self, orc: Oracle, h, bm):
        self.orc, self.h, self.bm = orc, h, bm
        L = orc._L
        self.n_rows = L.orc_plan_size(h, 0)
        self.n_tiles = L.orc_plan_size(h, 1)
        self.n_entries = L.orc_plan_size(h, 2)
        self.n_segs = L.orc_plan_size(h, 3)
        self.pairs = L.orc_plan_size(h, 4)
        z = lambda n: np.zeros(max(int(n), 1), dtype=np.int32)
        a = dict(seg_order=z(self.n_segs), seg_row_base=z(self.n_segs), row_pos=z(self.n_rows),
                 tile_seg=z(self.n_tiles), tile_t0=z(self.n_tiles), tile_rows=z(self.n_tiles),
                 tile_off=z(self.n_tiles + 1), entries=z(8 * self.n_entries),
                 csc_perm=z(self.n_entries), page_off=z(orc.num_pages + 1))
        L.orc_plan_arrays(h, *[_ip(a[k]) for k in ("seg_order", "seg_row_base", "row_pos", "tile_seg",
                                                     "tile_t0", "tile_rows", "tile_off", "entries",
                                                     "csc_perm", "page_off")])
        sizes = dict(seg_order=self.n_segs, seg_row_base=self.n_segs, row_pos=self.n_rows,
                     tile_seg=self.n_tiles, tile_t0=self.n_tiles, tile_rows=self.n_tiles,
                     tile_off=self.n_tiles + 1, entries=8 * self.n_entries, csc_perm=self.n_entries,
                     page_off=orc.num_pages + 1)
        for k, v in a.items():
            v = v[:sizes[k]]
            if k == "entries":
                v = v.reshape(-1, 8)
            setattr(self, k, v)

    def __del__(self):
        if getattr(self, "h", None):
            self.orc._L.orc_plan_delete(self.h)
            self.h = None

    def fwd(self, Q, scale, rows=None, nthreads=0):
        Q = np.ascontiguousarray(Q, dtype=np.float64)
        N, Hq, d = Q.shape
        assert N == self.n_rows
        O = np.zeros_like(Q)
        LSE = np.zeros((Hq, N), dtype=np.float64)
        r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
        st = self.orc._L.orc_fwd(self.h, Hq, _dp(Q), scale, _ip(r), -1 if r is None else len(r),
                                 _dp(O), _dp(LSE), nthreads)
        if st != OK:
            raise OracleError(st, "fwd")
        return O, LSE

    def bwd(self, Q, dO, scale, need_dq=None, need_dkdv=None, nthreads=0, partial=False):
        """Returns dQ [N,Hq,d] and dK, dV per token id [T,Hkv,d]."""
        Q = np.ascontiguousarray(Q, dtype=np.float64)
        dO = np.ascontiguousarray(dO, dtype=np.float64)
        N, Hq, d = Q.shape
        T = self.orc.n_tokens
        dQ = np.zeros_like(Q)
        dK = np.zeros((T, self.orc.Hkv, d))
        dV = np.zeros((T, self.orc.Hkv, d))
        nq = None if need_dq is None else np.ascontiguousarray(need_dq, dtype=np.uint8)
        nk = None if need_dkdv is None else np.ascontiguousarray(need_dkdv, dtype=np.uint8)
        st = self.orc._L.orc_bwd(self.h, Hq, _dp(Q), _dp(dO), scale, _up(nq), _up(nk),
                                 _dp(dQ), _dp(dK), _dp(dV), nthreads, 1 if partial else 0)
        if st != OK:
            raise OracleError(st, "bwd")
        return dQ, dK, dV

    def total_pairs(self):
        return int(self.orc._L.orc_plan_total_pairs(self.h))

    def row_context(self, r):
        n = self.orc._L.orc_row_context(self.h, r, None, None, 0)
        tok = np.zeros(max(n, 1), dtype=np.int32)
        src = np.zeros(max(n, 1), dtype=np.int32)
        self.orc._L.orc_row_context(self.h, r, _ip(tok), _ip(src), n)
        return tok[:n], src[:n]


def rope(x, pos, base, inverse=False):
    """Rotary embedding of x [n][H][d] (any float array; returned as a new fp64 array),
    row t at position pos[t] (orc_rope)."""
    L = _load()
    y = np.ascontiguousarray(np.array(x, dtype=np.float64))
    n, H, d = y.shape
    p = np.ascontiguousarray(np.asarray(pos, dtype=np.int32))
    assert p.shape == (n,)
    if L.orc_rope(_dp(y), n, H, d, _ip(p), float(base), 1 if inverse else 0):
        raise ValueError("orc_rope: bad arguments")
    return y
