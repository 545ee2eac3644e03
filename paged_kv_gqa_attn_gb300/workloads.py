"""Seeded synthetic inputs for paged GQA attention.

This module builds the inputs that both the CUDA path and the CPU oracle consume: the query
tensor, the paged K/V pools, the per-sequence block tables and the context lengths.  It holds
none of the attention arithmetic.  The fp8 pools are produced here by quantising N(0,1) data
with one symmetric scale per (physical block, kv head), which is how the workload is defined;
decoding those bytes back to numbers is left to each consumer.

Layouts (row-major, every tensor contiguous):
  q            [B, q_len, Hq, d]          bf16
  k/v cache    [num_blocks, Hkv, bs, d]   bf16, or uint8 holding fp8 E4M3 bit patterns
  k/v scale    [num_blocks, Hkv]          fp32 (fp8 only)
  block_table  [B, max_blocks_per_seq]    int32, -1 past each sequence's last block
  context_lens [B]                        int32, tokens in the cache including the q_len new ones

Block tables follow the PagedAttention description on the pages: the cache is cut into fixed
blocks of block_size tokens, each sequence owns an ordered list of logical blocks, and a table
maps each logical block to any physical block in a shared pool (studybook fde-roadmap ch.10,
section 10.4.2 "block table" and figure 10.4.2; aegloslab servingai 5.3.7).
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

KV_BF16 = "bf16"
KV_FP8_E4M3 = "fp8_e4m3"
FP8_E4M3_MAX = 448.0


@dataclasses.dataclass
class PagedAttnProblem:
    """One batch of paged-attention work, with everything the kernels and the oracle read."""

    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_table: torch.Tensor
    context_lens: torch.Tensor
    q_len: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    scale: float
    kv_dtype: str = KV_BF16
    k_scale: Optional[torch.Tensor] = None
    v_scale: Optional[torch.Tensor] = None
    name: str = "custom"
    seed: int = 0

    @property
    def num_seqs(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max().item()) if self.num_seqs else 0

    def to(self, device) -> "PagedAttnProblem":
        def mv(t):
            return None if t is None else t.to(device)

        return dataclasses.replace(
            self,
            q=mv(self.q),
            k_cache=mv(self.k_cache),
            v_cache=mv(self.v_cache),
            block_table=mv(self.block_table),
            context_lens=mv(self.context_lens),
            k_scale=mv(self.k_scale),
            v_scale=mv(self.v_scale),
        )


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def blocks_for(context_len: int, block_size: int) -> int:
    """Number of blocks a sequence of context_len tokens occupies (last one partly filled)."""
    return (int(context_len) + block_size - 1) // block_size


def allocate_block_tables(
    context_lens: Sequence[int],
    block_size: int,
    pool_factor: float = 1.25,
    free_fraction: Optional[float] = None,
    seed: int = 0,
    min_pool: int = 0,
):
    """Give every logical block of every sequence a distinct physical block, drawn at random.

    The pool holds ceil(need * pool_factor) blocks (or ceil(need / (1 - free_fraction)) when
    free_fraction is given).  A seeded permutation of the pool is walked in order; its first
    `need` entries are handed to the (sequence, logical block) pairs in sequence-major order, so
    the unused blocks end up interleaved at random positions of the pool.
    Returns (block_table int32 [B, max_blocks], num_blocks).
    """
    need_per_seq = [blocks_for(L, block_size) for L in context_lens]
    need = sum(need_per_seq)
    if free_fraction is not None:
        num_blocks = int(math.ceil(need / (1.0 - free_fraction)))
    else:
        num_blocks = int(math.ceil(need * pool_factor))
    num_blocks = max(num_blocks, need, min_pool, 1)
    perm = torch.randperm(num_blocks, generator=_gen(seed, "cpu")).to(torch.int32)
    max_blocks = max(max(need_per_seq) if need_per_seq else 1, 1)
    table = torch.full((len(context_lens), max_blocks), -1, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(need_per_seq):
        table[b, :n] = perm[pos : pos + n]
        pos += n
    return table, num_blocks


def _valid_slot_mask(block_table, context_lens, num_blocks, block_size):
    """[num_blocks, bs] bool: True where a physical slot holds a token of some sequence."""
    valid = torch.zeros(num_blocks, block_size, dtype=torch.bool)
    owned = torch.zeros(num_blocks, dtype=torch.bool)
    for b in range(block_table.shape[0]):
        L = int(context_lens[b])
        n = blocks_for(L, block_size)
        ids = block_table[b, :n].long()
        owned[ids] = True
        valid[ids] = True
        tail = L - (n - 1) * block_size
        if n > 0 and tail < block_size:
            valid[ids[n - 1], tail:] = False
    # blocks no sequence owns are treated as fully written (they are never read)
    valid[~owned] = True
    return valid


def quantize_fp8_e4m3(x: torch.Tensor, valid: torch.Tensor):
    """Quantise a pool [NB, Hkv, bs, d] to fp8 E4M3 with one scale per (block, kv head).

    scale = amax / 448 over the valid slots of that (block, head) tile (1 when amax is 0), the
    symmetric, zero-point-free scale quantisation of studybook fde-roadmap ch.10 section 10.8.2,
    with 448 the largest finite E4M3 value.  Slots that hold no token are zero-filled first.
    Returns (uint8 bit patterns, fp32 scales [NB, Hkv]).
    """
    x = x.float() * valid[:, None, :, None].to(x.device, torch.float32)
    amax = x.abs().amax(dim=(2, 3))
    scale = torch.where(amax > 0, amax / FP8_E4M3_MAX, torch.ones_like(amax)).to(torch.float32)
    q8 = (x / scale[:, :, None, None]).clamp(-FP8_E4M3_MAX, FP8_E4M3_MAX).to(torch.float8_e4m3fn)
    return q8.view(torch.uint8).contiguous(), scale.contiguous()


def make_problem(
    context_lens: Sequence[int],
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    block_size: int = 16,
    q_len: int = 1,
    kv_dtype: str = KV_BF16,
    pool_factor: float = 1.25,
    free_fraction: Optional[float] = None,
    min_pool: int = 0,
    scale: Optional[float] = None,
    seed: int = 0,
    device="cpu",
    tail_fill: str = "zero",
    name: str = "custom",
) -> PagedAttnProblem:
    """Build a seeded problem: Q, K, V ~ N(0,1) rounded to bf16 (or fp8 for the pools).

    tail_fill: "zero" leaves unused slots of partly filled blocks at 0; "nan" fills them (and
    every block no sequence owns) with NaN so that a kernel that reads past a context shows it.
    """
    B = len(context_lens)
    for L in context_lens:
        if L < 0:
            raise ValueError("context length must be >= 0")
    table, num_blocks = allocate_block_tables(
        context_lens, block_size, pool_factor, free_fraction, seed, min_pool
    )
    lens = torch.tensor(list(context_lens), dtype=torch.int32)
    gq = _gen(seed * 4 + 1, device)
    gk = _gen(seed * 4 + 2, device)
    gv = _gen(seed * 4 + 3, device)
    q = torch.randn(B, q_len, num_q_heads, head_dim, generator=gq, device=device).to(torch.bfloat16)
    shape = (num_blocks, num_kv_heads, block_size, head_dim)
    kf = torch.randn(*shape, generator=gk, device=device)
    vf = torch.randn(*shape, generator=gv, device=device)
    valid = _valid_slot_mask(table, lens, num_blocks, block_size)
    k_scale = v_scale = None
    if kv_dtype == KV_BF16:
        vm = valid.to(device)[:, None, :, None]
        if tail_fill == "nan":
            fill = torch.tensor(float("nan"), device=device)
        else:
            fill = torch.tensor(0.0, device=device)
        kc = torch.where(vm, kf, fill).to(torch.bfloat16)
        vc = torch.where(vm, vf, fill).to(torch.bfloat16)
        if tail_fill == "nan":
            owned = torch.zeros(num_blocks, dtype=torch.bool)
            for b in range(B):
                owned[table[b, : blocks_for(context_lens[b], block_size)].long()] = True
            un = (~owned).to(device)
            kc[un] = float("nan")
            vc[un] = float("nan")
    elif kv_dtype == KV_FP8_E4M3:
        kc, k_scale = quantize_fp8_e4m3(kf, valid.to(device))
        vc, v_scale = quantize_fp8_e4m3(vf, valid.to(device))
        if tail_fill == "nan":
            # 0x7F is the E4M3 NaN pattern
            vm = valid.to(device)[:, None, :, None].expand_as(kc)
            kc = torch.where(vm, kc, torch.full_like(kc, 0x7F))
            vc = torch.where(vm, vc, torch.full_like(vc, 0x7F))
    else:
        raise ValueError(f"unknown kv dtype {kv_dtype}")
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return PagedAttnProblem(
        q=q.contiguous(),
        k_cache=kc.contiguous(),
        v_cache=vc.contiguous(),
        block_table=table.to(device),
        context_lens=lens.to(device),
        q_len=q_len,
        num_q_heads=num_q_heads,
        num_kv_heads=num_kv_heads,
        head_dim=head_dim,
        block_size=block_size,
        scale=float(scale),
        kv_dtype=kv_dtype,
        k_scale=None if k_scale is None else k_scale.to(device),
        v_scale=None if v_scale is None else v_scale.to(device),
        name=name,
        seed=seed,
    )


# ---------------------------------------------------------------------------------------------
# Named workloads.  Shapes follow the serving set-up the pages discuss: an 8B GQA model with
# 32 query heads over 8 KV heads, head_dim 128, 2048-token contexts, 16-token blocks
# (aegloslab servingai 5.3.1 and 5.3.7), a continuous batch with ragged lengths (studybook
# fde-roadmap ch.10 section 10.5), speculative verify of K drafts plus one bonus position
# (sirzzang "Speculative Decoding" parallel verification) and an fp8 KV cache (section 10.8).
# ---------------------------------------------------------------------------------------------

BASE_SEED = 20261202

CONFIG_NAMES = (
    "tiny",
    "llama8b_decode",
    "cb_mix",
    "spec_verify_k4",
    "spec_verify_k8",
    "long_fp8",
    "llama70b_decode",
)


def config_context_lens(name: str, seed: int):
    """Context lengths (including new tokens) and q_len for a named workload."""
    g = _gen(seed * 4 + 0, "cpu")
    if name == "tiny":
        return [1, 17, 33, 64], 1
    if name == "llama8b_decode":
        return [2048] * 64, 1
    if name == "cb_mix":
        short = torch.randint(32, 513, (128,), generator=g)
        long = torch.randint(2048, 8193, (128,), generator=g)
        lens = torch.cat([short, long])
        order = torch.randperm(256, generator=g)
        return [int(x) for x in lens[order]], 1
    if name in ("spec_verify_k4", "spec_verify_k8"):
        K = 4 if name.endswith("4") else 8
        prior = torch.randint(1024, 4097, (16,), generator=g)
        return [int(x) + K + 1 for x in prior], K + 1
    if name == "long_fp8":
        return [131072] * 4, 1
    if name == "llama70b_decode":
        return [2048] * 64, 1
    raise KeyError(name)


def make_config(name: str, seed: Optional[int] = None, device="cpu", **overrides) -> PagedAttnProblem:
    """Build one of the named workloads with its default seed (BASE_SEED + workload index)."""
    idx = {"tiny": 0, "llama8b_decode": 1, "cb_mix": 2, "spec_verify_k4": 3,
           "spec_verify_k8": 3, "long_fp8": 4, "llama70b_decode": 5}[name]
    if seed is None:
        seed = BASE_SEED + idx
    lens, q_len = config_context_lens(name, seed)
    kw = dict(block_size=16, q_len=q_len, seed=seed, device=device, name=name)
    if name == "tiny":
        kw.update(num_q_heads=4, num_kv_heads=2, head_dim=64, min_pool=32, pool_factor=1.0)
    elif name == "llama70b_decode":
        kw.update(num_q_heads=64, num_kv_heads=8, head_dim=128)  # a group of 8 query heads
    else:
        kw.update(num_q_heads=32, num_kv_heads=8, head_dim=128)
    if name == "cb_mix":
        kw.update(free_fraction=0.10)
    if name == "long_fp8":
        kw.update(kv_dtype=KV_FP8_E4M3)
    kw.update(overrides)
    return make_problem(lens, **kw)


def random_tree_masks(num_seqs: int, q_len: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Ancestor bitmasks of random draft trees, int32 [B, q_len] (bit patterns of uint32).

    Node 0 is the root (the first new token); node t > 0 hangs under a random earlier node, so
    the nodes are in topological order.  Row t's mask has bit u set when u is t or one of its
    ancestors -- the tree form of speculative verification (aegloslab servingai 5.3.13).  A chain
    (every node under the previous one) gives the causal mask.
    """
    if q_len > 31:
        raise ValueError("tree masks here hold at most 31 new tokens")
    g = _gen(seed * 4 + 3, "cpu")
    masks = torch.zeros(num_seqs, q_len, dtype=torch.int64)
    for b in range(num_seqs):
        for t in range(q_len):
            if t == 0:
                masks[b, t] = 1
            else:
                parent = int(torch.randint(0, t, (1,), generator=g))
                masks[b, t] = masks[b, parent] | (1 << t)
    return masks.to(torch.int32).to(device)


def chain_mask(num_seqs: int, q_len: int, device="cpu") -> torch.Tensor:
    """The causal mask as ancestor bitmasks: row t sees new tokens 0..t."""
    row = torch.tensor([(1 << (t + 1)) - 1 for t in range(q_len)], dtype=torch.int64)
    return row.expand(num_seqs, q_len).contiguous().to(torch.int32).to(device)


# ---------------------------------------------------------------------------------------------
# Inputs of the speculative acceptance step (the distributions a verify round produces)

LLAMA3_VOCAB = 128256


@dataclasses.dataclass
class AcceptProblem:
    """One round of speculative acceptance for a batch: target probabilities at the K + 1
    verified positions, draft probabilities at the K drafted positions, the drafted tokens, and
    the uniforms the round consumes."""

    p: torch.Tensor          # [B, K+1, V] fp32
    q: torch.Tensor          # [B, K, V] fp32
    draft: torch.Tensor      # [B, K] int32
    u_accept: torch.Tensor   # [B, K] fp32 in [0, 1)
    u_sample: torch.Tensor   # [B] int32 holding uint32 bit patterns

    @property
    def num_seqs(self) -> int:
        return int(self.p.shape[0])

    @property
    def num_draft(self) -> int:
        return int(self.q.shape[1])

    @property
    def vocab(self) -> int:
        return int(self.p.shape[2])

    def to(self, device) -> "AcceptProblem":
        return AcceptProblem(*(t.to(device) for t in (self.p, self.q, self.draft, self.u_accept, self.u_sample)))


def make_accept_problem(num_seqs: int, num_draft: int, vocab: int, seed: int = 0, device="cpu",
                        target_temp: float = 3.0, draft_noise: float = 1.0) -> AcceptProblem:
    """Target logits ~ N(0, target_temp^2) per position; draft logits = target logits + N(0,
    draft_noise^2) (a draft that roughly agrees with the target); both turned into probabilities
    with torch's softmax in fp32; each draft token drawn from its q row with torch.multinomial;
    uniforms from the same seeded generator.  The last target position has no draft."""
    g = _gen(seed, "cpu")
    z = torch.randn(num_seqs, num_draft + 1, vocab, generator=g) * target_temp
    zq = z[:, :num_draft] + torch.randn(num_seqs, num_draft, vocab, generator=g) * draft_noise
    p = torch.softmax(z, dim=-1).float()
    q = torch.softmax(zq, dim=-1).float()
    if num_draft:
        draft = torch.multinomial(q.reshape(-1, vocab), 1, generator=g).reshape(num_seqs, num_draft)
    else:
        draft = torch.zeros(num_seqs, 0, dtype=torch.int64)
    u_accept = torch.rand(num_seqs, num_draft, generator=g).float()
    words = torch.randint(0, 2 ** 32, (num_seqs,), generator=g, dtype=torch.int64)
    u_sample = (words - (words >= 2 ** 31).long() * 2 ** 32).to(torch.int32)  # same bits as uint32
    return AcceptProblem(p.contiguous(), q.contiguous(), draft.to(torch.int32).contiguous(),
                         u_accept.contiguous(), u_sample.contiguous()).to(device)


ACCEPT_CONFIGS = {
    # the verify shapes' batches with the Llama-3 vocabulary
    "spec_accept_k4": (16, 4, LLAMA3_VOCAB),
    "spec_accept_k8": (16, 8, LLAMA3_VOCAB),
    "spec_accept_b256_k4": (256, 4, LLAMA3_VOCAB),
}


def make_accept_config(name: str, seed: Optional[int] = None, device="cpu") -> AcceptProblem:
    B, K, V = ACCEPT_CONFIGS[name]
    return make_accept_problem(B, K, V, seed=BASE_SEED + 100 + list(ACCEPT_CONFIGS).index(name)
                               if seed is None else seed, device=device)


# ---------------------------------------------------------------------------------------------
# Packed variable-length query rows (chunked prefill with piggybacked decode / verify rows)


@dataclasses.dataclass
class VarlenProblem:
    """A batch whose sequences bring different numbers of new rows: sequence b's q_len_b rows
    are q[query_start_loc[b]:query_start_loc[b+1]], and context_lens[b] = prior_b + q_len_b."""

    q: torch.Tensor                # [total_q, Hq, d] bf16
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_table: torch.Tensor
    context_lens: torch.Tensor
    query_start_loc: torch.Tensor  # [B + 1] int32
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    scale: float
    kv_dtype: str = KV_BF16
    k_scale: Optional[torch.Tensor] = None  # [num_blocks, Hkv] fp32 (E4M3 caches)
    v_scale: Optional[torch.Tensor] = None

    @property
    def num_seqs(self) -> int:
        return int(self.block_table.shape[0])

    @property
    def q_lens(self):
        qsl = self.query_start_loc.cpu().tolist()
        return [qsl[i + 1] - qsl[i] for i in range(len(qsl) - 1)]

    @property
    def max_q_len(self) -> int:
        return max(self.q_lens) if self.num_seqs else 1

    def to(self, device) -> "VarlenProblem":
        return dataclasses.replace(self, q=self.q.to(device), k_cache=self.k_cache.to(device),
                                   v_cache=self.v_cache.to(device), block_table=self.block_table.to(device),
                                   context_lens=self.context_lens.to(device),
                                   query_start_loc=self.query_start_loc.to(device),
                                   k_scale=None if self.k_scale is None else self.k_scale.to(device),
                                   v_scale=None if self.v_scale is None else self.v_scale.to(device))


def make_varlen_problem(prior_lens: Sequence[int], q_lens: Sequence[int], num_q_heads: int,
                        num_kv_heads: int, head_dim: int, seed: int = 0, device="cpu",
                        tail_fill: str = "zero", pool_factor: float = 1.25,
                        kv_dtype: str = KV_BF16) -> VarlenProblem:
    """Caches and tables as make_problem for contexts prior + q_len (the new rows' K/V already
    appended; bf16, or E4M3 with per-(block, kv head) scales); packed queries N(0, 1) rounded to
    bf16."""
    if len(prior_lens) != len(q_lens):
        raise ValueError("prior_lens and q_lens differ in length")
    lens = [int(a) + int(n) for a, n in zip(prior_lens, q_lens)]
    base = make_problem(lens, num_q_heads, num_kv_heads, head_dim, seed=seed, device=device,
                        tail_fill=tail_fill, pool_factor=pool_factor, kv_dtype=kv_dtype)
    qsl = [0]
    for n in q_lens:
        qsl.append(qsl[-1] + int(n))
    g = _gen(seed * 4 + 5, device)
    q = torch.randn(qsl[-1], num_q_heads, head_dim, generator=g, device=device).to(torch.bfloat16)
    return VarlenProblem(q.contiguous(), base.k_cache, base.v_cache, base.block_table, base.context_lens,
                         torch.tensor(qsl, dtype=torch.int32, device=device), num_q_heads, num_kv_heads,
                         head_dim, base.block_size, base.scale, kv_dtype=base.kv_dtype, k_scale=base.k_scale,
                         v_scale=base.v_scale)


def chunked_prefill_workload(seed: Optional[int] = None, device="cpu", chunk: int = 512,
                             num_seqs: int = 4, decodes: int = 0, kv_dtype: str = KV_BF16) -> VarlenProblem:
    """Chunked prefill of the Llama-3-8B attention shape: num_seqs prompts whose chunk of `chunk`
    new tokens follows a prior context drawn U[0, 4096] (earlier chunks already cached), plus
    `decodes` piggybacked decode rows with contexts U[1024, 4096]; KV bf16 or E4M3."""
    s = BASE_SEED + 200 if seed is None else seed
    g = torch.Generator().manual_seed(s)
    prior = torch.randint(0, 4097, (num_seqs,), generator=g).tolist()
    qls = [chunk] * num_seqs
    if decodes:
        prior += torch.randint(1023, 4096, (decodes,), generator=g).tolist()
        qls += [1] * decodes
    return make_varlen_problem(prior, qls, 32, 8, 128, seed=s, device=device, kv_dtype=kv_dtype)
