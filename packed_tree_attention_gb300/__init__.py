"""packed_tree_attention_gb300 -- Python binding of liboctopus (include/octopus.h).

Argument marshalling only: every step of the hot path (the tile-list compiler, the
attention forward/backward and the paged decode) runs in the library's CUDA kernels.
There is no CPU fallback: importing works without a GPU, but any call that needs the
device fails loudly if the CUDA library or a GPU is missing.

Names follow the C ABI: ``Pool.fork`` is ``octo_fork``, ``Plan.attn_fwd`` is
``octo_attn_fwd`` and so on; the module-level ``octo_*`` aliases take the same
arguments as the C functions' Python counterparts.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = _build.LIB

OK, EINVAL, ENOMEM, ESTATE, ECUDA, ETIMEOUT, ENOTSUP, ESCRATCH = range(8)
NOALLOC_SCRATCH_BYTES = 32 << 20
DTYPE_F32, DTYPE_BF16 = 0, 1

_lib = None


class OctoError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = _lib.octo_strerror(code).decode() if _lib is not None else str(code)
        extra = ""
        if code == ECUDA and _lib is not None:
            extra = " (cudaError %d)" % _lib.octo_last_cuda_error()
        super().__init__(f"{what}: {msg}{extra} [status {code}]")
        self.code = code


class _Desc(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32), ("k_pool", ctypes.c_void_p),
                ("v_pool", ctypes.c_void_p)]


class _SegInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("parent", "fork", "len", "n_pages", "refcount", "p_next", "flags")]


class _PoolState(ctypes.Structure):
    _fields_ = [("n_segments", ctypes.c_int32), ("free_pages", ctypes.c_int32), ("n_mounts", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("seg_capacity", ctypes.c_int32),
                ("refcount", ctypes.POINTER(ctypes.c_int32)), ("n_pages", ctypes.POINTER(ctypes.c_int32)),
                ("page_owner", ctypes.POINTER(ctypes.c_int32))]


class _PlanInfo(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int64), ("n_tiles", ctypes.c_int64), ("n_entries", ctypes.c_int64),
                ("n_segments", ctypes.c_int64), ("pairs", ctypes.c_int64), ("bm", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_tile_entries", ctypes.c_int32),
                ("max_page_entries", ctypes.c_int32), ("n_touched_pages", ctypes.c_int32),
                ("is_decode", ctypes.c_int32), ("n_rec_runs", ctypes.c_int32), ("n_rec_chunks", ctypes.c_int32)]


ENTRY_DTYPE = np.dtype([("q_tile", "<u4"), ("kv_page", "<u4"), ("kv_lo", "<u2"), ("kv_hi", "<u2"),
                        ("q_lo", "<u2"), ("flags", "<u2"), ("diag", "<i4"), ("src", "<i4")])
assert ENTRY_DTYPE.itemsize == 24

# exported symbols of include/octopus.h
SYMBOLS = ("octo_pool_create", "octo_pool_destroy", "octo_root", "octo_append", "octo_fork", "octo_mount",
           "octo_rewind", "octo_done", "octo_unpin", "octo_release", "octo_pool_info", "octo_seg_query",
           "octo_pack_tree", "octo_decode_plan", "octo_plan_info", "octo_plan_copy_out", "octo_plan_destroy",
           "octo_attn_fwd", "octo_attn_bwd_workspace_size", "octo_attn_bwd", "octo_decode_workspace_size",
           "octo_decode", "octo_strerror", "octo_last_cuda_error", "octo_sync", "octo_kernel_path",
           "octo_launch_count", "octo_decode_noalloc", "octo_append_rope", "octo_rope_rows",
           "octo_rope_pool_grad", "octo_token_logprob_workspace_size", "octo_token_logprob",
           "octo_decode_plan_advance", "octo_pool_query", "octo_decode_cursors", "octo_recurrent_workspace_size",
           "octo_recurrent_fwd", "octo_recurrent_bwd", "octo_wait_selftest", "octo_append_step")


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Loads liboctopus.so (building it with nvcc if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing:
        _build.build()
    if not os.path.exists(LIB_PATH):
        raise ImportError("liboctopus.so is not built; run packed_tree_attention_gb300/build.py")
    L = ctypes.CDLL(LIB_PATH)
    I32, P, IP = ctypes.c_int32, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)
    SZ = ctypes.c_size_t
    F = ctypes.c_float
    sig = {
        "octo_pool_create": [ctypes.POINTER(_Desc), ctypes.POINTER(P)],
        "octo_pool_destroy": [P],
        "octo_root": [P, IP],
        "octo_append": [P, I32, I32, P, P, P, IP],
        "octo_fork": [P, I32, I32, IP],
        "octo_mount": [P, I32, I32, I32, I32, IP],
        "octo_rewind": [P, I32, I32, IP],
        "octo_done": [P, I32],
        "octo_unpin": [P, I32],
        "octo_release": [P, I32],
        "octo_pool_info": [P, IP, IP, IP],
        "octo_seg_query": [P, I32, ctypes.POINTER(_SegInfo), IP, IP],
        "octo_pack_tree": [P, IP, I32, I32, P, ctypes.POINTER(P)],
        "octo_decode_plan": [P, IP, I32, P, ctypes.POINTER(P)],
        "octo_plan_info": [P, ctypes.POINTER(_PlanInfo)],
        "octo_plan_copy_out": [P] + [P] * 10,
        "octo_plan_destroy": [P],
        "octo_attn_fwd": [P, I32, P, P, P, P, P, F, P],
        "octo_attn_bwd_workspace_size": [P, I32],
        "octo_attn_bwd": [P, I32, P, P, P, P, P, P, P, P, P, F, P, SZ, P],
        "octo_decode_workspace_size": [P, I32],
        "octo_decode": [P, I32, P, P, P, P, P, F, P, SZ, P],
        "octo_strerror": [ctypes.c_int],
        "octo_last_cuda_error": [],
        "octo_sync": [P, P],
        "octo_kernel_path": [P, I32, I32],
        "octo_launch_count": [],
        "octo_decode_noalloc": [P, I32, P, P, P, P, P, F, P],
        "octo_append_rope": [P, I32, I32, P, P, F, P, IP],
        "octo_rope_rows": [P, I32, P, I32, F, I32, P],
        "octo_rope_pool_grad": [P, P, F, P],
        "octo_token_logprob_workspace_size": [I32, ctypes.POINTER(SZ)],
        "octo_token_logprob": [P, I32, I32, P, I32, ctypes.c_int64, I32, P, P, P, P, P, F, P, P, SZ, P],
        "octo_decode_plan_advance": [P, P],
        "octo_pool_query": [P, ctypes.POINTER(_PoolState)],
        "octo_decode_cursors": [P, IP, I32, I32, P, P, P, P, P, F, P, SZ, P],
        "octo_recurrent_workspace_size": [P, I32, I32],
        "octo_wait_selftest": [P, ctypes.c_uint32, P],
        "octo_append_step": [P, IP, I32, P, P, F, P, IP],
        "octo_recurrent_fwd": [P, I32, I32, P, P, P, P, P, P, P, SZ, P],
        "octo_recurrent_bwd": [P, I32, I32, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    L.octo_strerror.restype = ctypes.c_char_p
    L.octo_attn_bwd_workspace_size.restype = SZ
    L.octo_decode_workspace_size.restype = SZ
    L.octo_recurrent_workspace_size.restype = SZ
    L.octo_launch_count.argtypes = []
    L.octo_launch_count.restype = ctypes.c_int64
    _lib = L
    return L


def launch_count() -> int:
    """Kernels the library has enqueued in this process so far (octo_launch_count)."""
    return int(load().octo_launch_count())


def _ptr(x):
    """Address of a tensor argument.  The library reads plain pointers with the dense
    layouts its header gives, so a view with gaps or reordered strides is refused here
    rather than read wrongly."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError("tensor arguments must be contiguous (got strides %s for shape %s)"
                         % (tuple(x.stride()), tuple(x.shape)))
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _chk(st, what):
    if st != OK:
        raise OctoError(st, what)


def _ip(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


class Pool:
    """A paged, refcounted KV pool and its episode DAG (octo_pool_create)."""

    def __init__(self, num_pages, page_size, n_kv_heads, head_dim, dtype, k_pool=None, v_pool=None):
        L = load()
        self._L = L
        self.num_pages, self.page_size, self.n_kv_heads, self.head_dim = num_pages, page_size, n_kv_heads, head_dim
        self.dtype = dtype
        self.k_pool, self.v_pool = k_pool, v_pool      # keep the caller's tensors alive
        d = _Desc(num_pages, page_size, n_kv_heads, head_dim, dtype, _ptr(k_pool), _ptr(v_pool))
        h = ctypes.c_void_p()
        _chk(L.octo_pool_create(ctypes.byref(d), ctypes.byref(h)), "octo_pool_create")
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            self._L.octo_pool_destroy(self.h)
            self.h = None

    __del__ = close

    def root(self):
        out = ctypes.c_int32()
        _chk(self._L.octo_root(self.h, ctypes.byref(out)), "octo_root")
        return out.value

    def append(self, cur, n, k=None, v=None, stream=None, check=True):
        pos = np.zeros(max(n, 1), dtype=np.int32)
        st = self._L.octo_append(self.h, cur, n, _ptr(k), _ptr(v), _stream(stream), _ip(pos))
        if not check:
            return st
        _chk(st, "octo_append")
        return pos[:n]

    def append_rope(self, cur, n, k, v, base, stream=None, check=True):
        """octo_append_rope: append with the K rows rotated at the positions they receive."""
        pos = np.zeros(max(n, 1), dtype=np.int32)
        st = self._L.octo_append_rope(self.h, cur, n, _ptr(k), _ptr(v), float(base), _stream(stream), _ip(pos))
        if not check:
            return st
        _chk(st, "octo_append_rope")
        return pos[:n]

    def append_step(self, cursors, k=None, v=None, rope_base=0.0, stream=None, check=True):
        """octo_append_step: one token for each of the (distinct) cursors in one call."""
        c = np.ascontiguousarray(cursors, dtype=np.int32)
        pos = np.zeros(max(len(c), 1), dtype=np.int32)
        st = self._L.octo_append_step(self.h, _ip(c), len(c), _ptr(k), _ptr(v), float(rope_base), _stream(stream),
                                      _ip(pos))
        if not check:
            return st
        _chk(st, "octo_append_step")
        return pos[:len(c)]

    def fork(self, cur, n, check=True):
        out = np.zeros(max(n, 1), dtype=np.int32)
        st = self._L.octo_fork(self.h, cur, n, _ip(out))
        if not check:
            return st
        _chk(st, "octo_fork")
        return out[:n].tolist()

    def mount(self, reader, producer, a, b, check=True):
        out = ctypes.c_int32()
        st = self._L.octo_mount(self.h, reader, producer, a, b, ctypes.byref(out))
        if not check:
            return st
        _chk(st, "octo_mount")
        return out.value

    def rewind(self, cur, k, check=True):
        out = ctypes.c_int32()
        st = self._L.octo_rewind(self.h, cur, k, ctypes.byref(out))
        if not check:
            return st
        _chk(st, "octo_rewind")
        return out.value

    def done(self, cur, check=True):
        st = self._L.octo_done(self.h, cur)
        if check:
            _chk(st, "octo_done")
        return st

    def unpin(self, cur, check=True):
        st = self._L.octo_unpin(self.h, cur)
        if check:
            _chk(st, "octo_unpin")
        return st

    def release(self, cur, check=True):
        st = self._L.octo_release(self.h, cur)
        if check:
            _chk(st, "octo_release")
        return st

    def info(self):
        a, b, c = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _chk(self._L.octo_pool_info(self.h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)), "octo_pool_info")
        return dict(n_segments=a.value, free_pages=b.value, n_mounts=c.value)

    def query(self):
        """octo_pool_query: counts, every segment's refcount and page count, and the owner
        of every page (-1 free)."""
        n = self.info()["n_segments"]
        rc = np.zeros(max(n, 1), dtype=np.int32)
        npg = np.zeros(max(n, 1), dtype=np.int32)
        own = np.zeros(self.num_pages, dtype=np.int32)
        st = _PoolState(0, 0, 0, 0, len(rc), _ip(rc), _ip(npg), _ip(own))
        _chk(self._L.octo_pool_query(self.h, ctypes.byref(st)), "octo_pool_query")
        return dict(n_segments=st.n_segments, free_pages=st.free_pages, n_mounts=st.n_mounts,
                    num_pages=st.num_pages, refcount=rc[:st.n_segments], n_pages=npg[:st.n_segments],
                    page_owner=own)

    def decode_cursors(self, cursors, n_q_heads, q, out, lse, scale, ws=None, ws_bytes=None, k_pool=None,
                       v_pool=None, stream=None):
        """octo_decode_cursors: plan, decode and plan release in one call (ws None: the
        library takes the workspace from the stream-ordered allocator)."""
        c = np.ascontiguousarray(cursors, dtype=np.int32)
        if ws_bytes is None:
            ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
        _chk(self._L.octo_decode_cursors(self.h, _ip(c), len(c), n_q_heads, _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                         _ptr(out), _ptr(lse), float(scale), _ptr(ws), ws_bytes, _stream(stream)),
             "octo_decode_cursors")

    def seg_info(self, s):
        i = _SegInfo()
        _chk(self._L.octo_seg_query(self.h, s, ctypes.byref(i), None, None), "octo_seg_query")
        return {n: getattr(i, n) for n, _ in _SegInfo._fields_}

    def seg_pos(self, s):
        n = self.seg_info(s)["len"]
        out = np.zeros(max(n, 1), dtype=np.int32)
        _chk(self._L.octo_seg_query(self.h, s, None, _ip(out), None), "octo_seg_query")
        return out[:n]

    def seg_pages(self, s):
        n = self.seg_info(s)["n_pages"]
        out = np.zeros(max(n, 1), dtype=np.int32)
        _chk(self._L.octo_seg_query(self.h, s, None, None, _ip(out)), "octo_seg_query")
        return out[:n]

    def pack_tree(self, roots, bm, stream=None):
        r = np.ascontiguousarray(roots, dtype=np.int32)
        h = ctypes.c_void_p()
        _chk(self._L.octo_pack_tree(self.h, _ip(r), len(r), bm, _stream(stream), ctypes.byref(h)), "octo_pack_tree")
        return Plan(self, h)

    def decode_plan(self, cursors, stream=None):
        c = np.ascontiguousarray(cursors, dtype=np.int32)
        h = ctypes.c_void_p()
        _chk(self._L.octo_decode_plan(self.h, _ip(c), len(c), _stream(stream), ctypes.byref(h)), "octo_decode_plan")
        return Plan(self, h)


class Plan:
    """A compiled block-sparse schedule (octo_pack_tree / octo_decode_plan)."""

    def __init__(self, pool: Pool, h):
        self.pool, self._L, self.h = pool, pool._L, h
        self.info = self._info()

    def _info(self):
        i = _PlanInfo()
        _chk(self._L.octo_plan_info(self.h, ctypes.byref(i)), "octo_plan_info")
        return {n: getattr(i, n) for n, _ in _PlanInfo._fields_}

    def close(self):
        if getattr(self, "h", None):
            self._L.octo_plan_destroy(self.h)
            self.h = None

    __del__ = close

    def copy_out(self):
        I = self.info
        z = lambda n: np.zeros(max(int(n), 1), dtype=np.int32)
        a = dict(seg_order=z(I["n_segments"]), seg_row_base=z(I["n_segments"]), row_pos=z(I["n_rows"]),
                 tile_seg=z(I["n_tiles"]), tile_t0=z(I["n_tiles"]), tile_rows=z(I["n_tiles"]),
                 tile_off=z(I["n_tiles"] + 1), csc_perm=z(I["n_entries"]), page_off=z(self.pool.num_pages + 1))
        ent = np.zeros(max(I["n_entries"], 1), dtype=ENTRY_DTYPE)
        p = lambda x: x.ctypes.data
        _chk(self._L.octo_plan_copy_out(self.h, p(a["seg_order"]), p(a["seg_row_base"]), p(a["row_pos"]),
                                        p(a["tile_seg"]), p(a["tile_t0"]), p(a["tile_rows"]), p(a["tile_off"]),
                                        p(ent), p(a["csc_perm"]), p(a["page_off"])), "octo_plan_copy_out")
        n = dict(seg_order=I["n_segments"], seg_row_base=I["n_segments"], row_pos=I["n_rows"],
                 tile_seg=I["n_tiles"], tile_t0=I["n_tiles"], tile_rows=I["n_tiles"], tile_off=I["n_tiles"] + 1,
                 csc_perm=I["n_entries"], page_off=self.pool.num_pages + 1)
        out = {k: v[:n[k]] for k, v in a.items()}
        out["entries"] = ent[:I["n_entries"]]
        return out

    def attn_fwd(self, n_q_heads, q, o, lse, scale, k_pool=None, v_pool=None, stream=None):
        _chk(self._L.octo_attn_fwd(self.h, n_q_heads, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(o), _ptr(lse),
                                   float(scale), _stream(stream)), "octo_attn_fwd")

    def attn_bwd_workspace_size(self, n_q_heads):
        return int(self._L.octo_attn_bwd_workspace_size(self.h, n_q_heads))

    def attn_bwd(self, n_q_heads, q, o, lse, dout, dq, dk_pool, dv_pool, scale, ws, ws_bytes=None, k_pool=None,
                 v_pool=None, stream=None):
        if ws_bytes is None:
            ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
        _chk(self._L.octo_attn_bwd(self.h, n_q_heads, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(o), _ptr(lse),
                                   _ptr(dout), _ptr(dq), _ptr(dk_pool), _ptr(dv_pool), float(scale), _ptr(ws),
                                   ws_bytes, _stream(stream)), "octo_attn_bwd")

    def decode_workspace_size(self, n_q_heads):
        return int(self._L.octo_decode_workspace_size(self.h, n_q_heads))

    def decode(self, n_q_heads, q, out, lse, scale, ws=None, ws_bytes=None, k_pool=None, v_pool=None, stream=None):
        if ws_bytes is None:
            ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
        _chk(self._L.octo_decode(self.h, n_q_heads, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(out), _ptr(lse),
                                 float(scale), _ptr(ws), ws_bytes, _stream(stream)), "octo_decode")

    def decode_noalloc(self, n_q_heads, q, out, lse, scale, k_pool=None, v_pool=None, stream=None):
        """octo_decode_noalloc: the decode without a workspace argument, for callers that
        cannot allocate device memory (its partials use the library's static scratch)."""
        _chk(self._L.octo_decode_noalloc(self.h, n_q_heads, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(out),
                                         _ptr(lse), float(scale), _stream(stream)), "octo_decode_noalloc")

    def rope_rows(self, n_heads, x, base, inverse=False, stream=None):
        """octo_rope_rows: rotate the plan's packed rows of x (bf16 or fp32) in place."""
        dt = DTYPE_F32 if x.element_size() == 4 else DTYPE_BF16
        _chk(self._L.octo_rope_rows(self.h, n_heads, _ptr(x), dt, float(base), 1 if inverse else 0, _stream(stream)),
             "octo_rope_rows")

    def rope_pool_grad(self, dk_pool, base, stream=None):
        """octo_rope_pool_grad: key gradients back through the append rotation."""
        _chk(self._L.octo_rope_pool_grad(self.h, _ptr(dk_pool), float(base), _stream(stream)), "octo_rope_pool_grad")

    def advance(self, stream=None, check=True):
        """octo_decode_plan_advance: the decode plan one token further on every cursor."""
        st = self._L.octo_decode_plan_advance(self.h, _stream(stream))
        if st == OK:
            self.info = self._info()
        if check:
            _chk(st, "octo_decode_plan_advance")
        return st

    def token_logprob_workspace_size(self, n_rows):
        n = ctypes.c_size_t(0)
        _chk(self._L.octo_token_logprob_workspace_size(n_rows, ctypes.byref(n)), "octo_token_logprob_workspace_size")
        return n.value

    def token_logprob(self, row0, n_rows, logits, vocab, ids, weight, logp, ws, row_lse=None, dlogits=None,
                      grad_scale=1.0, loss=None, stream=None):
        """octo_token_logprob: per-token log-probabilities (and loss, gradient) of the rows
        [row0, row0 + n_rows) whose logits rows are `logits` [n_rows][ld] (bf16 or fp32)."""
        dt = DTYPE_F32 if logits.element_size() == 4 else DTYPE_BF16
        _chk(self._L.octo_token_logprob(self.h, row0, n_rows, _ptr(logits), dt, logits.stride(0), vocab,
                                        _ptr(ids), _ptr(weight), _ptr(logp), _ptr(row_lse), _ptr(dlogits),
                                        float(grad_scale), _ptr(loss), _ptr(ws), ws.numel() * ws.element_size(),
                                        _stream(stream)), "octo_token_logprob")

    def recurrent_workspace_size(self, n_heads, head_dim):
        return int(self._L.octo_recurrent_workspace_size(self.h, n_heads, head_dim))

    def recurrent_fwd(self, n_heads, head_dim, q, k, v, alpha, beta, o, ws, stream=None):
        """octo_recurrent_fwd: the gated delta rule over the packed rows (fp32); ws keeps what
        the backward needs."""
        _chk(self._L.octo_recurrent_fwd(self.h, n_heads, head_dim, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                                        _ptr(beta), _ptr(o), _ptr(ws), ws.numel() * ws.element_size(),
                                        _stream(stream)), "octo_recurrent_fwd")

    def recurrent_bwd(self, n_heads, head_dim, q, k, v, alpha, beta, dout, dq, dk, dv, dalpha, dbeta, ws,
                      stream=None):
        """octo_recurrent_bwd: gradients of octo_recurrent_fwd (same inputs and workspace)."""
        _chk(self._L.octo_recurrent_bwd(self.h, n_heads, head_dim, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                                        _ptr(beta), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dalpha),
                                        _ptr(dbeta), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
             "octo_recurrent_bwd")

    def sync(self, stream=None):
        _chk(self._L.octo_sync(self.h, _stream(stream)), "octo_sync")

    def wait_selftest(self, max_polls, stream=None):
        """octo_wait_selftest: a bounded device wait that expires (OCTO_ETIMEOUT at the next sync)."""
        _chk(self._L.octo_wait_selftest(self.h, max_polls, _stream(stream)), "octo_wait_selftest")

    def kernel_path(self, n_q_heads, which):
        return int(self._L.octo_kernel_path(self.h, n_q_heads, which))


# module-level aliases with the C names
def octo_pool_create(num_pages, page_size, n_kv_heads, head_dim, dtype, k_pool=None, v_pool=None):
    return Pool(num_pages, page_size, n_kv_heads, head_dim, dtype, k_pool, v_pool)


def octo_pack_tree(pool, roots, bm, stream=None):
    return pool.pack_tree(roots, bm, stream)


def octo_decode_plan(pool, cursors, stream=None):
    return pool.decode_plan(cursors, stream)


def octo_attn_fwd(plan, n_q_heads, q, o, lse, scale, k_pool=None, v_pool=None, stream=None):
    return plan.attn_fwd(n_q_heads, q, o, lse, scale, k_pool, v_pool, stream)


def octo_attn_bwd(plan, n_q_heads, q, o, lse, dout, dq, dk_pool, dv_pool, scale, ws, ws_bytes=None, k_pool=None,
                  v_pool=None, stream=None):
    return plan.attn_bwd(n_q_heads, q, o, lse, dout, dq, dk_pool, dv_pool, scale, ws, ws_bytes, k_pool, v_pool,
                         stream)


def octo_decode(plan, n_q_heads, q, out, lse, scale, ws=None, ws_bytes=None, k_pool=None, v_pool=None, stream=None):
    return plan.decode(n_q_heads, q, out, lse, scale, ws, ws_bytes, k_pool, v_pool, stream)
