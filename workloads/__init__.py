"""Seeded synthetic inputs for one paged-KV decode step.

Test and benchmark infrastructure.  Both the CPU oracle (``oracle/``) and the
CUDA library are fed from the arrays built here; this module holds none of the
attention arithmetic and imports neither side.

What it builds, per workload:

* ``seq_lens``      int32 [B]     lengths *after* this step's append (the query of
                                 sequence s attends over positions [0, L_s)).
* ``block_tables``  int32 [B, W]  logical -> physical block ids; entries past a
                                 sequence's last block are poison ids that no
                                 kernel may dereference.
* pools             uint16 bit patterns [NB, bs, Hkv, d] of fp16 / bf16, one K
                                 and one V pool per layer.  Slots that hold no
                                 token before the step are NaN.  An 8-bit
                                 (E4M3) pool holds uint8 codes drawn at random
                                 over a few binades, with per-layer, per-KV-head
                                 float32 scales (``k_scales`` / ``v_scales``).
* ``q``             [B, Hq, d];  ``k_new`` / ``v_new`` [T, Hkv, d] with
  ``slot_mapping`` int64 [T] (slot < 0: padding entry, nothing is written).
* ``copy_pairs``    int64 [Np, 2] (src, dst) copy-on-write pairs for a fork.

The allocation (which physical block backs which logical block) is drawn the
way the pages' host block managers hand blocks out: a free list that is a
seeded permutation of the pool, consumed in order ("LLM 推理引擎内部原理" §2.3
``BlockEngine``; tbr8.org PagedAttention article §3 ``BlockManager``).  The
slot of a token is the flat index ``physical_block * block_size + offset``
that ``BlockEngine.append_slot`` returns (same page, §2.3).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

F16 = "f16"
BF16 = "bf16"
E4M3 = "e4m3"
DTYPES = (F16, BF16)
# quiet-NaN bit patterns used to poison slots that hold no token
NAN_BITS = {F16: 0x7E00, BF16: 0x7FC0}
E4M3_NAN = 0x7F
INT32_MAX = np.iinfo(np.int32).max


# --------------------------------------------------------------------------
# dtype encoding of the random values (input plumbing, not the method)
# --------------------------------------------------------------------------
def f32_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to fp16 / bf16 (nearest-even) and return the uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        u = x.view(np.uint32)
        lsb = (u >> np.uint32(16)) & np.uint32(1)
        return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    raise ValueError(dtype)


def random_e4m3_codes(rng: np.random.Generator, shape) -> np.ndarray:
    """Random finite 8-bit E4M3 codes: random sign, exponent field 4..9
    (magnitudes 2^-3 .. 7.5), random mantissa.  Arbitrary cache bytes, not a
    quantization of anything."""
    n = int(np.prod(shape))
    sign = rng.integers(0, 2, n, dtype=np.uint8) << 7
    exp = rng.integers(4, 10, n, dtype=np.uint8) << 3
    man = rng.integers(0, 8, n, dtype=np.uint8)
    return (sign | exp | man).reshape(shape)


def normal_bits(rng: np.random.Generator, shape, dtype: str, chunk: int = 1 << 24) -> np.ndarray:
    """N(0,1) samples drawn as float32 from ``rng`` and rounded to ``dtype`` bits."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        out[lo:hi] = f32_to_bits(rng.standard_normal(hi - lo, dtype=np.float32), dtype)
    return out.reshape(shape)


# --------------------------------------------------------------------------
# workload specifications
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class Spec:
    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str
    seed: int
    lens: tuple              # ("fixed", (...)) | ("uniform", lo, hi) | ("lognormal", median, sigma, lo, hi) | ("const", L)
    pool: tuple = ("headroom", 0.2)   # ("fixed", NB) | ("headroom", fraction)
    num_layers: int = 1
    fork: tuple | None = None         # (requests, n, prefix_len, suffix_lo, suffix_hi)
    description: str = ""
    kv_dtype: str = ""                # "" = the pool holds `dtype`; E4M3 = 8-bit codes with scales

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads

    @property
    def elem_bytes(self) -> int:
        """Bytes of a q / out / new K-V element (fp16 or bf16)."""
        return 2

    @property
    def fp8(self) -> bool:
        return self.kv_dtype == E4M3

    @property
    def kv_elem_bytes(self) -> int:
        """Bytes of a pool element."""
        return 1 if self.fp8 else 2


SPECS = {
    "tiny": Spec(
        "tiny", 4, 4, 4, 64, 16, F16, 1001, ("fixed", (1, 17, 33, 50)), ("fixed", 32),
        description="4 seqs {1,17,33,50}, 4 q / 4 kv heads, d64, bs16, fp16, permuted pool of 32"),
    "llama3_8b": Spec(
        "llama3_8b", 64, 32, 8, 128, 16, BF16, 1002, ("uniform", 512, 4096),
        description="Llama-3-8B-shaped layer: 64 seqs U[512,4096], 32 q / 8 kv heads, d128, bs16, bf16, pool +20%"),
    "llama3_8b_fp8": Spec(
        "llama3_8b_fp8", 64, 32, 8, 128, 16, BF16, 1006, ("uniform", 512, 4096), kv_dtype=E4M3,
        description="as llama3_8b with an 8-bit E4M3 K/V pool (per-KV-head scales), bf16 q and out"),
    "llama2_70b_mixed_bs16": Spec(
        "llama2_70b_mixed_bs16", 128, 64, 8, 128, 16, F16, 1003, ("lognormal", 500.0, 1.2, 32, 8192),
        description="Llama-2-70B-shaped layer: 128 seqs lognormal(500,1.2) in [32,8192], 64 q / 8 kv, d128, bs16, fp16"),
    "llama2_70b_mixed_bs32": Spec(
        "llama2_70b_mixed_bs32", 128, 64, 8, 128, 32, F16, 1003, ("lognormal", 500.0, 1.2, 32, 8192),
        description="as llama2_70b_mixed_bs16 at block_size 32 (same lengths, its own pool)"),
    "cow_fork": Spec(
        "cow_fork", 768, 32, 8, 128, 8, F16, 1004, ("fork",), num_layers=1,
        fork=(256, 3, 1024, 0, 512),
        description="256 requests x n=3 forks sharing a 1024-token prefix, suffix U[0,512], 32 q / 8 kv, d128, bs8, fp16"),
    "cow_fork_partial": Spec(
        "cow_fork_partial", 768, 32, 8, 128, 8, F16, 1042, ("fork",), num_layers=1,
        fork=(256, 3, 1020, 0, 512),
        description="as cow_fork with a 1020-token prefix (last prefix block half filled)"),
    "llama2_70b_step": Spec(
        "llama2_70b_step", 16, 64, 8, 128, 16, BF16, 1005, ("const", 4096), ("headroom", 0.0), num_layers=80,
        description="Llama-2-70B decode step: 80 layers x (append + decode), 16 seqs at 4096, 64 q / 8 kv, d128, bs16, bf16"),
}


def small_spec(**kw) -> Spec:
    """A custom spec for edge-case tests (defaults: one layer, fp16, bs16)."""
    base = dict(name="custom", num_seqs=3, num_heads=8, num_kv_heads=2, head_dim=128,
                block_size=16, dtype=F16, seed=7, lens=("fixed", (5, 40, 17)), pool=("headroom", 0.5))
    base.update(kw)
    return Spec(**base)


# --------------------------------------------------------------------------
# host block allocator (harness; the pages' free-list manager)
# --------------------------------------------------------------------------
class BlockAllocator:
    """Free list over a pool of ``num_blocks`` physical blocks.

    The free list is ``rng.permutation(num_blocks)`` consumed front to back, so
    physically adjacent blocks are rarely logically adjacent.  ``allocate``
    returns None when the pool is exhausted, as the pages' managers do.
    """

    def __init__(self, num_blocks: int, rng: np.random.Generator):
        self.free = [int(b) for b in rng.permutation(num_blocks)]
        self.pos = 0

    def allocate(self, n: int):
        if self.pos + n > len(self.free):
            return None
        out = self.free[self.pos:self.pos + n]
        self.pos += n
        return out


def blocks_needed(num_tokens: int, block_size: int) -> int:
    return -(-num_tokens // block_size)


# --------------------------------------------------------------------------
# the built workload
# --------------------------------------------------------------------------
@dataclass
class Workload:
    spec: Spec
    num_blocks: int
    seq_lens: np.ndarray            # int32 [B]
    block_tables: np.ndarray        # int32 [B, W]
    q: np.ndarray                   # uint16 [B, Hq, d]
    k_new: np.ndarray               # uint16 [T, Hkv, d]
    v_new: np.ndarray               # uint16 [T, Hkv, d]
    slot_mapping: np.ndarray        # int64 [T]
    copy_pairs: np.ndarray          # int64 [Np, 2]
    valid_slots: np.ndarray         # bool [NB, bs]: slots holding a token before the step
    key_caches: list = field(default_factory=list)    # per layer uint16 (uint8 for E4M3) [NB, bs, Hkv, d]
    value_caches: list = field(default_factory=list)
    layer_seeds: list = field(default_factory=list)
    k_scales: list = field(default_factory=list)      # per layer float32 [Hkv] (E4M3 pools only)
    v_scales: list = field(default_factory=list)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.spec.head_dim)

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if len(self.seq_lens) else 0

    @property
    def num_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])

    def pool_shape(self):
        s = self.spec
        return (self.num_blocks, s.block_size, s.num_kv_heads, s.head_dim)

    def pool_bytes_per_layer(self) -> int:
        """Bytes of one layer's K pool plus V pool."""
        return 2 * int(np.prod(self.pool_shape())) * self.spec.kv_elem_bytes


def _draw_lens(spec: Spec, rng: np.random.Generator) -> np.ndarray:
    kind = spec.lens[0]
    B = spec.num_seqs
    if kind == "fixed":
        v = np.array(spec.lens[1], dtype=np.int64)
    elif kind == "uniform":
        v = rng.integers(spec.lens[1], spec.lens[2], endpoint=True, size=B)
    elif kind == "lognormal":
        med, sigma, lo, hi = spec.lens[1:]
        v = np.clip(np.rint(rng.lognormal(mean=math.log(med), sigma=sigma, size=B)), lo, hi)
    elif kind == "const":
        v = np.full(B, spec.lens[1], dtype=np.int64)
    else:
        raise ValueError(kind)
    assert v.shape == (B,)
    return v.astype(np.int64)


def build(spec: Spec, values: str = "host") -> Workload:
    """Build the inputs of one decode step of ``spec``.

    ``values``: "host" draws every pool value with numpy on the host; "none"
    builds only the structure (tables, lengths, slots, pairs, q and new k/v)
    and leaves the pools to ``device_pools`` (used for the 80-layer workload).
    """
    rng = np.random.default_rng(spec.seed)
    bs = spec.block_size
    B = spec.num_seqs

    # ---- lengths, appended positions and block tables ------------------------
    if spec.fork is None:
        lens = _draw_lens(spec, rng)
        need = sum(blocks_needed(int(L), bs) for L in lens)
        if spec.pool[0] == "fixed":
            NB = int(spec.pool[1])
        else:
            NB = int(math.ceil(need * (1.0 + spec.pool[1])))
        assert need <= NB
        alloc = BlockAllocator(NB, rng)
        tables = [alloc.allocate(blocks_needed(int(L), bs)) for L in lens]
        # one new token per sequence at position L-1 (lengths are post-append)
        appended = [[int(L) - 1] if L > 0 else [] for L in lens]
        cow_pairs = []
        cow_dst = set()
    else:
        reqs, n, P, lo, hi = spec.fork
        assert reqs * n == B
        sfx = rng.integers(lo, hi, endpoint=True, size=(reqs, n))
        lens = (P + sfx).reshape(-1).astype(np.int64)
        nbp = blocks_needed(P, bs)
        Pc = nbp * bs
        need = reqs * nbp + reqs * (n - 1)
        for L in lens:
            need += max(0, blocks_needed(int(L), bs) - nbp)
        NB = int(math.ceil(need * (1.0 + spec.pool[1])))
        alloc = BlockAllocator(NB, rng)
        tables, appended, cow_pairs, cow_dst = [], [], [], set()
        for r in range(reqs):
            prefix = alloc.allocate(nbp)
            for f in range(n):
                L = int(lens[r * n + f])
                t = list(prefix)
                if f > 0:
                    # copy-on-write of the last prefix block for every fork but the first
                    dst = alloc.allocate(1)[0]
                    cow_pairs.append((t[-1], dst))
                    cow_dst.add(dst)
                    t[-1] = dst
                t += alloc.allocate(max(0, blocks_needed(L, bs) - nbp))
                tables.append(t)
                # positions written by this step: the rest of the (copied) last prefix
                # block, and the newest token
                pos = set(range(P, min(L, Pc)))
                if L > P:
                    pos.add(L - 1)
                appended.append(sorted(pos))

    W = max(1, max(len(t) for t in tables))
    bt = np.empty((B, W), dtype=np.int64)
    # poison padding: alternate an id just past the pool and INT32_MAX
    bt[:, 0::2] = NB + 7
    bt[:, 1::2] = INT32_MAX
    for s, t in enumerate(tables):
        bt[s, :len(t)] = t
    block_tables = bt.astype(np.int32)

    # ---- slots valid before the step ----------------------------------------
    valid = np.zeros((NB, bs), dtype=bool)
    for s in range(B):
        t = np.asarray(tables[s], dtype=np.int64)
        L = int(lens[s])
        pre = np.ones(L, dtype=bool)
        if appended[s]:
            pre[np.asarray(appended[s])] = False
        pos = np.nonzero(pre)[0]
        blk = t[pos // bs] if len(pos) else pos
        keep = np.array([int(b) not in cow_dst for b in blk], dtype=bool) if cow_dst else np.ones(len(pos), bool)
        valid[blk[keep], (pos % bs)[keep]] = True

    # ---- appended tokens -----------------------------------------------------
    slots = []
    for s in range(B):
        t = tables[s]
        if not appended[s]:
            slots.append(-1)      # padding entry: sequence appends nothing this step
        for p in appended[s]:
            slots.append(int(t[p // bs]) * bs + p % bs)
    slot_mapping = np.asarray(slots, dtype=np.int64)
    T = len(slots)

    Hq, Hkv, d = spec.num_heads, spec.num_kv_heads, spec.head_dim
    q = normal_bits(rng, (B, Hq, d), spec.dtype)
    k_new = normal_bits(rng, (T, Hkv, d), spec.dtype)
    v_new = normal_bits(rng, (T, Hkv, d), spec.dtype)

    wl = Workload(spec=spec, num_blocks=NB, seq_lens=lens.astype(np.int32), block_tables=block_tables,
                  q=q, k_new=k_new, v_new=v_new, slot_mapping=slot_mapping,
                  copy_pairs=np.asarray(cow_pairs, dtype=np.int64).reshape(-1, 2), valid_slots=valid)
    wl.layer_seeds = [int(spec.seed) * 1000 + l for l in range(spec.num_layers)]
    if spec.fp8:
        # per-KV-head scales of each layer, so dequantized codes are O(1)
        srng = np.random.default_rng((spec.seed, 8))
        for _ in range(spec.num_layers):
            wl.k_scales.append(srng.uniform(0.05, 0.3, Hkv).astype(np.float32))
            wl.v_scales.append(srng.uniform(0.05, 0.3, Hkv).astype(np.float32))
    if values == "host":
        for l in range(spec.num_layers):
            lrng = np.random.default_rng(wl.layer_seeds[l])
            if spec.fp8:
                kc = random_e4m3_codes(lrng, wl.pool_shape())
                vc = random_e4m3_codes(lrng, wl.pool_shape())
                nan = np.uint8(E4M3_NAN)
            else:
                kc = normal_bits(lrng, wl.pool_shape(), spec.dtype)
                vc = normal_bits(lrng, wl.pool_shape(), spec.dtype)
                nan = np.uint16(NAN_BITS[spec.dtype])
            kc[~valid] = nan
            vc[~valid] = nan
            wl.key_caches.append(kc)
            wl.value_caches.append(vc)
    elif values != "none":
        raise ValueError(values)
    return wl


def device_pools(wl: Workload, layer: int, device="cuda"):
    """One layer's K and V pools drawn directly on the device (torch generator).

    Used where host generation would take minutes (the 80-layer workload).  The
    values are N(0,1) rounded to the pool dtype, unused slots NaN; a test reads
    back the blocks it checks.
    """
    import torch

    spec = wl.spec
    g = torch.Generator(device=device)
    g.manual_seed(wl.layer_seeds[layer])
    mask = torch.from_numpy(~wl.valid_slots).to(device)
    out = []
    for _ in range(2):
        if spec.fp8:                               # random finite E4M3 codes, as random_e4m3_codes
            shape = wl.pool_shape()
            sign = torch.randint(0, 2, shape, generator=g, device=device, dtype=torch.uint8) << 7
            exp = torch.randint(4, 10, shape, generator=g, device=device, dtype=torch.uint8) << 3
            man = torch.randint(0, 8, shape, generator=g, device=device, dtype=torch.uint8)
            x = sign | exp | man
            x[mask] = E4M3_NAN
        else:
            tdt = torch.float16 if spec.dtype == F16 else torch.bfloat16
            x = torch.randn(wl.pool_shape(), generator=g, device=device, dtype=torch.float32).to(tdt)
            x[mask] = float("nan")
        out.append(x)
    return out[0], out[1]


def host_pools_for(wl: Workload, seqs, layer: int = 0):
    """One layer's host pools with values only in the blocks ``seqs`` use (rest NaN).

    For timing the CPU oracle on a sample without drawing the whole pool.
    Values come from a generator seeded by (layer seed, block id), so a block's
    contents do not depend on which sample asked for it.
    """
    spec = wl.spec
    if spec.fp8:
        nan, store = np.uint8(E4M3_NAN), np.uint8
        draw = lambda rng, shape: random_e4m3_codes(rng, shape)
    else:
        nan, store = np.uint16(NAN_BITS[spec.dtype]), np.uint16
        draw = lambda rng, shape: normal_bits(rng, shape, spec.dtype)
    kc = np.full(wl.pool_shape(), nan, dtype=store)
    vc = np.full(wl.pool_shape(), nan, dtype=store)
    blk_shape = wl.pool_shape()[1:]
    for s in seqs:
        nb = blocks_needed(int(wl.seq_lens[s]), spec.block_size)
        for b in wl.block_tables[s, :nb]:
            b = int(b)
            rng = np.random.default_rng((wl.layer_seeds[layer], b))
            kc[b] = draw(rng, blk_shape)
            vc[b] = draw(rng, blk_shape)
            kc[b][~wl.valid_slots[b]] = nan
            vc[b][~wl.valid_slots[b]] = nan
    return kc, vc
