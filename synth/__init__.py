"""Seeded synthetic inputs shared by the oracle tests, the CUDA path tests and bench.py.

This module holds none of the method's arithmetic: no positions, masks, tile lists,
softmax or packing.  It only emits

* episode op logs -- sequences of the pool primitives (root / append / fork /
  mount / rewind / done / release / unpin) whose shapes follow the episode
  statistics quoted on the Octopus project page ("Architecture & Co-Design",
  the primitives table, and the "Emergent Collective Scaling" figures), and
* random tensors (K/V rows per appended token, Q/dO rows per segment token,
  decode queries) drawn from numpy's PCG64 and rounded once to the stored dtype.

The small amount of bookkeeping kept here (lengths, parents, which producer was
already mounted on a lineage) is used only to choose ops that the pool accepts.

Cursor ids equal segment ids: the n-th segment created by root/fork/rewind gets
id n, on both the oracle and the library side.
"""
from __future__ import annotations

import dataclasses
import numpy as np

__all__ = ["Episode", "CONFIGS", "make_preset", "random_dag", "round_bf16",
           "bf16_bits", "bits_to_f32", "Tensors", "make_tensors", "make_decode_q"]


# --------------------------------------------------------------------------------------
# op log
# --------------------------------------------------------------------------------------
class Episode:
    """An op log plus the structural bookkeeping needed to keep it valid."""

    def __init__(self, page_size: int):
        self.page_size = page_size
        self.ops: list[tuple] = []
        self.parent: list[int] = []
        self.length: list[int] = []
        self.appendable: list[bool] = []
        self.mounted: set[tuple[int, int]] = set()   # (reader segment, producer segment)
        self.roots: list[int] = []
        self.cursors: list[int] = []      # cursors a decode step queries (decode presets)
        self.n_tokens = 0

    # -- primitives -------------------------------------------------------------------
    def _new(self, parent: int) -> int:
        self.parent.append(parent)
        self.length.append(0)
        self.appendable.append(True)
        return len(self.parent) - 1

    def root(self) -> int:
        self.ops.append(("root",))
        s = self._new(-1)
        self.roots.append(s)
        return s

    def append(self, c: int, n: int) -> None:
        assert self.appendable[c] and n >= 0
        if n == 0:
            return
        self.ops.append(("append", c, n))
        self.length[c] += n
        self.n_tokens += n

    def fork(self, c: int, n: int) -> list[int]:
        assert self.appendable[c] and n >= 1
        self.ops.append(("fork", c, n))
        return [self._new(c) for _ in range(n)]

    def rewind(self, c: int, k: int) -> int:
        assert self.appendable[c] and 0 <= k <= self.length[c]
        self.ops.append(("rewind", c, k))
        self.appendable[c] = False
        return self._new(c)

    def done(self, c: int) -> None:
        self.ops.append(("done", c))
        self.appendable[c] = False

    def lineage(self, c: int) -> list[int]:
        out = []
        while c >= 0:
            out.append(c)
            c = self.parent[c]
        return out

    def can_mount(self, r: int, p: int) -> bool:
        """Conservative structural check: the producer is not on the reader's lineage,
        and no segment on the reader's lineage mounted this producer before."""
        lin = self.lineage(r)
        if p in lin or not self.appendable[r]:
            return False
        return not any((x, p) in self.mounted for x in lin)

    def mount(self, r: int, p: int, a: int, b: int, checked: bool = True) -> None:
        """checked=False records a mount that can_mount's conservative rule would refuse
        (an ancestor's tokens past the fork point, a second span of a producer already
        mounted on the lineage); the caller has made sure the pool accepts it."""
        assert 0 <= a < b <= self.length[p] and self.appendable[r]
        assert not checked or self.can_mount(r, p)
        self.ops.append(("mount", r, p, a, b))
        self.mounted.add((r, p))

    @property
    def n_segments(self) -> int:
        return len(self.parent)


# --------------------------------------------------------------------------------------
# configurations (heads, dims, page size, dtype, value scale)
# --------------------------------------------------------------------------------------
CONFIGS = {
    # tiny fp32 tree: 1 head, d=64, page 16
    "tiny": dict(Hq=1, Hkv=1, d=64, P=16, dtype="f32", scale=1.0),
    # bf16 single tree, forward only
    "tree_fwd": dict(Hq=16, Hkv=4, d=128, P=64, dtype="bf16", scale=0.5),
    # bf16 full episode, forward + backward
    "episode": dict(Hq=16, Hkv=4, d=128, P=64, dtype="bf16", scale=0.5),
    # bf16 training step over 8 trees, forward + backward
    "train_step": dict(Hq=16, Hkv=4, d=128, P=64, dtype="bf16", scale=0.5),
    # the first tree of the training step alone (the small case of its ncu captures)
    "train_tree": dict(Hq=16, Hkv=4, d=128, P=64, dtype="bf16", scale=0.5),
    # paged decode, 256 cursors
    "decode": dict(Hq=16, Hkv=4, d=128, P=64, dtype="bf16", scale=0.5),
    # the same cursor shape, 4 episodes x 8 cursors (about 1 GB of K/V: profiling runs)
    "decode_small": dict(Hq=16, Hkv=4, d=128, P=64, dtype="bf16", scale=0.5),
}


def _tiny() -> Episode:
    """Prefix of 64 tokens forked into two branches of 32; branch B (16 tokens in)
    mounts span [8, 24) of branch A, then appends its last 16 tokens."""
    ep = Episode(16)
    r = ep.root()
    ep.append(r, 64)
    a, b = ep.fork(r, 2)
    ep.append(a, 32)
    ep.append(b, 16)
    ep.mount(b, a, 8, 24)
    ep.append(b, 16)
    return ep


def _tree_fwd() -> Episode:
    """4K prefix forked into 4 branches of 8K; branch 1 reads branch 0 [0, 2048) and
    branch 3 reads branch 2 [4096, 6144), both after 4096 own tokens."""
    ep = Episode(64)
    r = ep.root()
    ep.append(r, 4096)
    b = ep.fork(r, 4)
    ep.append(b[0], 8192)
    ep.append(b[2], 8192)
    ep.append(b[1], 4096)
    ep.mount(b[1], b[0], 0, 2048)
    ep.append(b[1], 4096)
    ep.append(b[3], 4096)
    ep.mount(b[3], b[2], 4096, 6144)
    ep.append(b[3], 4096)
    return ep


def _episode(seed: int) -> Episode:
    """16K prefix, 7 branches that each own 32K tokens (dead-end leaves included),
    3 rewinds leaving dead leaves of 1-4K, 6 sibling mounts of 1-8K tokens."""
    rng = np.random.default_rng(np.random.PCG64(seed))
    ep = Episode(64)
    r = ep.root()
    ep.append(r, 16384)
    branches = ep.fork(r, 7)
    budget = 32768
    cur = list(branches)            # current cursor of each branch
    owned = [0] * 7
    rew = set(rng.choice(7, size=3, replace=False).tolist())
    rew_at = {i: int(rng.integers(2048, budget - 8192)) for i in rew}
    rew_len = {i: int(rng.integers(1024, 4097)) for i in rew}
    rewound = set()
    n_mounts, want_mounts = 0, 6
    chunk = 1024
    # mount times: after this many round-robin rounds
    rounds = budget // chunk
    mount_rounds = sorted(rng.choice(np.arange(3, rounds - 1), size=want_mounts, replace=False).tolist())
    for rd in range(rounds + 8):
        for i in range(7):
            if owned[i] >= budget:
                continue
            n = min(chunk, budget - owned[i])
            if i in rew and i not in rewound and owned[i] + n > rew_at[i]:
                # grow to the rewind point plus a detour, then rewind: the detour stays
                # as a dead-end leaf
                pre = rew_at[i] - owned[i]
                ep.append(cur[i], pre)
                ep.append(cur[i], rew_len[i])
                k = ep.length[cur[i]] - rew_len[i]
                cur[i] = ep.rewind(cur[i], k)
                owned[i] += pre + rew_len[i]
                rewound.add(i)
                continue
            ep.append(cur[i], n)
            owned[i] += n
        while n_mounts < want_mounts and mount_rounds and mount_rounds[0] <= rd:
            mount_rounds.pop(0)
            for _ in range(64):
                ri, pi = rng.choice(7, size=2, replace=False).tolist()
                rc, pc = cur[ri], cur[pi]
                if owned[ri] >= budget or not ep.can_mount(rc, pc) or ep.length[pc] < 1024:
                    continue
                span = int(rng.integers(1024, 8193))
                span = min(span, ep.length[pc])
                a = int(rng.integers(0, ep.length[pc] - span + 1))
                ep.mount(rc, pc, a, a + span)
                n_mounts += 1
                break
        if all(o >= budget for o in owned):
            break
    return ep


def _train_step(seed: int, n_trees: int = 8, target: int = 140_000) -> Episode:
    """8 random trees: root prefix, fork fan-out 2-6 per level, depth <= 3, branch
    growth <= 32K, 0-4 mounts per reader of 0.5-8K, each tree 140K owned tokens (1.12M
    in all)."""
    rng = np.random.default_rng(np.random.PCG64(seed))
    ep = Episode(64)
    for _ in range(n_trees):
        _random_tree(ep, rng, target)
    return ep


def _random_tree(ep: Episode, rng, target: int) -> None:
    r = ep.root()
    prefix = int(rng.integers(2048, 8193))
    ep.append(r, prefix)
    total = prefix
    # plan: list of (cursor, depth) leaves to grow; grow breadth-first
    frontier = [(r, 0)]
    leaves = []
    while frontier:
        c, depth = frontier.pop(0)
        if depth >= 3 or total >= target:
            leaves.append(c)
            continue
        k = int(rng.integers(2, 7))
        kids = ep.fork(c, k)
        for kid in kids:
            remaining = target - total
            if remaining <= 0:
                leaves.append(kid)
                continue
            grow = int(rng.integers(512, 32769))
            # keep room for deeper levels
            grow = min(grow, max(1, remaining // max(1, k)))
            ep.append(kid, grow)
            total += grow
            if depth + 1 < 3 and rng.random() < 0.5 and total < target:
                frontier.append((kid, depth + 1))
            else:
                leaves.append(kid)
    # 0-4 mounts per reader leaf, spans of 0.5-8K from non-lineage segments of this tree,
    # each followed by a few of the reader's own tokens
    leaves = [c for c in leaves if ep.appendable[c]]
    tree_segs = [s for s in range(r, ep.n_segments)]
    for c in leaves:
        nm = int(rng.integers(0, 5))
        for _ in range(nm):
            cands = [p for p in tree_segs if p != c and ep.length[p] >= 512 and ep.can_mount(c, p)]
            if not cands:
                break
            p = cands[int(rng.integers(0, len(cands)))]
            span = min(int(rng.integers(512, 8193)), ep.length[p])
            a = int(rng.integers(0, ep.length[p] - span + 1))
            ep.mount(c, p, a, a + span)
            n = min(int(rng.integers(64, 1025)), max(0, target - total))
            ep.append(c, n)
            total += n
    # then top the leaves up round-robin until the tree owns exactly `target` tokens
    li = 0
    while total < target and leaves:
        c = leaves[li % len(leaves)]
        n = min(int(rng.integers(512, 4097)), target - total)
        ep.append(c, n)
        total += n
        li += 1


def _decode(seed: int, n_episodes: int = 32, per_episode: int = 8) -> Episode:
    """32 episodes x 8 cursors: a shared prefix of 2-8K, each cursor's path 8-32K,
    0-3 mounted sibling spans of 0.5-8K, then the one token that is decoded."""
    rng = np.random.default_rng(np.random.PCG64(seed))
    ep = Episode(64)
    for _ in range(n_episodes):
        r = ep.root()
        prefix = int(rng.integers(2048, 8193))
        ep.append(r, prefix)
        kids = ep.fork(r, per_episode)
        for k in kids:
            path = int(rng.integers(8192, 32769))
            ep.append(k, max(1, path - prefix))
        for k in kids:
            nm = int(rng.integers(0, 4))
            sibs = [s for s in kids if s != k]
            rng.shuffle(sibs)
            for p in sibs[:nm]:
                span = min(int(rng.integers(512, 8193)), ep.length[p])
                a = int(rng.integers(0, ep.length[p] - span + 1))
                ep.mount(k, p, a, a + span)
        for k in kids:
            ep.append(k, 1)          # the token whose query is decoded
        ep.cursors.extend(kids)
    return ep


def random_dag(seed: int, page_size: int = 16, max_segments: int = 12,
               max_len: int = 80, p_mount: float = 0.5, p_rewind: float = 0.3,
               p_done: float = 0.2, n_roots: int = 1) -> Episode:
    """Small random episodes for bit-exact and parity tests: random fork fan-out,
    ragged lengths (zero-length segments included), rewinds, mounts between any
    non-lineage segments, done/pins."""
    rng = np.random.default_rng(np.random.PCG64(seed))
    ep = Episode(page_size)
    for _ in range(n_roots):
        r = ep.root()
        ep.append(r, int(rng.integers(0, max_len)))
    live = list(range(ep.n_segments))
    steps = 0
    while ep.n_segments < max_segments * n_roots and steps < 200:
        steps += 1
        live = [c for c in live if ep.appendable[c]]
        if not live:
            break
        c = live[int(rng.integers(0, len(live)))]
        u = rng.random()
        if u < 0.35:
            ep.append(c, int(rng.integers(1, max_len)))
        elif u < 0.55:
            kids = ep.fork(c, int(rng.integers(1, 4)))
            for kid in kids:
                ep.append(kid, int(rng.integers(0, max_len)))
            live.extend(kids)
        elif u < 0.55 + 0.45 * p_mount:
            cands = [p for p in range(ep.n_segments) if ep.length[p] > 0 and ep.can_mount(c, p)]
            if cands:
                p = cands[int(rng.integers(0, len(cands)))]
                a = int(rng.integers(0, ep.length[p]))
                b = int(rng.integers(a + 1, ep.length[p] + 1))
                ep.mount(c, p, a, b)
                ep.append(c, int(rng.integers(0, max_len // 2 + 1)))
        elif u < 0.55 + 0.45 * p_mount + 0.45 * p_rewind:
            if ep.length[c] > 0:
                k = int(rng.integers(0, ep.length[c] + 1))
                n = ep.rewind(c, k)
                ep.append(n, int(rng.integers(0, max_len)))
                live.append(n)
        elif rng.random() < p_done:
            ep.done(c)
    return ep


def make_preset(name: str, seed: int = 0) -> Episode:
    if name == "tiny":
        return _tiny()
    if name == "tree_fwd":
        return _tree_fwd()
    if name == "episode":
        return _episode(seed)
    if name == "train_step":
        return _train_step(seed)
    if name == "train_tree":
        return _train_step(seed, n_trees=1)
    if name == "decode":
        return _decode(seed)
    if name == "decode_small":
        return _decode(seed, n_episodes=4)
    raise KeyError(name)


# --------------------------------------------------------------------------------------
# tensors
# --------------------------------------------------------------------------------------
def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    u = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return u.view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 values that are bf16-representable -> their uint16 bit patterns."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _draw(rng, shape, scale, dtype):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return round_bf16(x) if dtype == "bf16" else x


@dataclasses.dataclass
class Tensors:
    """K/V rows per token in append order [T, Hkv, d]; Q/dO rows per segment token,
    segments in id order [sum(len), Hq, d] with seg_off[s] the first row of segment s.
    Values are float32 arrays holding exactly the stored (bf16 or fp32) values."""
    K: np.ndarray
    V: np.ndarray
    Q: np.ndarray
    dO: np.ndarray
    seg_off: np.ndarray
    dtype: str


def make_tensors(ep: Episode, Hq: int, Hkv: int, d: int, dtype: str, scale: float,
                 seed: int, with_do: bool = True) -> Tensors:
    rng = np.random.default_rng(np.random.PCG64(seed + 0x5EED))
    T = ep.n_tokens
    K = _draw(rng, (T, Hkv, d), scale, dtype)
    V = _draw(rng, (T, Hkv, d), scale, dtype)
    seg_off = np.zeros(ep.n_segments + 1, dtype=np.int64)
    seg_off[1:] = np.cumsum(ep.length)
    N = int(seg_off[-1])
    Q = _draw(rng, (N, Hq, d), scale, dtype)
    dO = _draw(rng, (N, Hq, d), 1.0, dtype) if with_do else None
    return Tensors(K, V, Q, dO, seg_off, dtype)


def make_decode_q(n: int, Hq: int, d: int, dtype: str, scale: float, seed: int) -> np.ndarray:
    rng = np.random.default_rng(np.random.PCG64(seed + 0xDEC0DE))
    return _draw(rng, (n, Hq, d), scale, dtype)


# --------------------------------------------------------------------------------------
# counter-based generator for large workloads
# --------------------------------------------------------------------------------------
# Large benchmark tensors (hundreds of millions of values) are drawn from a counter-based
# generator so that the GPU can fill them in place while the CPU side evaluates exactly
# the same values for the few rows it checks.  Element e of stream s is
#     x = (sum of twelve 16-bit uniforms) / 65536 - 6
# (the classic twelve-uniform approximation of a unit normal: mean 0, variance 1), the
# uniforms taken from the MurmurHash3 32-bit finalizer applied to (s, e, k).  Only
# integer operations and exact power-of-two scalings are involved, so torch on any
# device produces identical bits; values are then scaled by a power of two and rounded
# to the stored dtype.

_M32 = 0xFFFFFFFF
_GOLD = 0x9E3779B9


def _mul32(h, c):
    lo = h & 0xFFFF
    hi = h >> 16
    return (lo * c + ((hi * (c & 0xFFFF)) << 16)) & _M32


def _fmix32(h):
    h = h ^ (h >> 16)
    h = _mul32(h, 0x85EBCA6B)
    h = h ^ (h >> 13)
    h = _mul32(h, 0xC2B2AE35)
    return h ^ (h >> 16)


def hash_normal(stream: int, index, scale: float = 1.0):
    """Values of stream `stream` at int64 element indices `index` (a torch tensor on any
    device).  Returns float32 (scale must be a power of two for bit-identity)."""
    import torch
    e = index.to(torch.int64)
    seed = ((stream * _GOLD) ^ 0x5BD1E995) & _M32
    base = _fmix32((e & _M32) ^ _fmix32(((e >> 32) + seed) & _M32))
    acc = torch.zeros_like(e)
    for k in range(6):
        u = _fmix32((base + (k + 1) * _GOLD) & _M32)
        acc = acc + (u & 0xFFFF) + (u >> 16)
    x = (acc - 6 * 65536).to(torch.float32) * (1.0 / 65536.0)
    return x * scale


def hash_fill(stream: int, shape, dtype, device, scale: float = 1.0, row_start: int = 0, chunk_rows: int = 65536):
    """A tensor of `shape` whose flat element i holds hash_normal(stream, row_start *
    row_size + i) * scale, rounded to dtype.  Filled in row chunks to bound memory."""
    import torch
    out = torch.empty(shape, dtype=dtype, device=device)
    rows = shape[0]
    row_size = 1
    for s in shape[1:]:
        row_size *= s
    flat = out.view(rows, row_size)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        idx = torch.arange((row_start + r0) * row_size, (row_start + r1) * row_size, device=device,
                           dtype=torch.int64)
        flat[r0:r1] = hash_normal(stream, idx, scale).view(r1 - r0, row_size).to(dtype)
    return out


def hash_rows(stream: int, rows, row_size: int, dtype, scale: float = 1.0, device="cpu"):
    """Values of selected rows (numpy int array of row ids) of a hash_fill tensor, as a
    numpy float64 array [len(rows), row_size] holding the dtype-rounded values; computed
    on `device` (identical bits on any device)."""
    import torch
    r = torch.as_tensor(np.asarray(rows, dtype=np.int64)).to(device)
    idx = (r[:, None] * row_size + torch.arange(row_size, dtype=torch.int64, device=device)[None, :]).reshape(-1)
    x = hash_normal(stream, idx, scale).to(dtype).to(torch.float64)
    return x.view(len(rows), row_size).cpu().numpy()


STREAM_K, STREAM_V, STREAM_Q, STREAM_DO, STREAM_DECODE_Q = 1, 2, 3, 4, 5
