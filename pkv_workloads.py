"""Seeded synthetic workloads for the paged-KV path: decode steps (plain, GQA,
shared prefixes, FP8, beam search), chunked-prefill steps, prompts that share a
system prompt (prefix caching) and swap steps.

This module only draws random numbers and lays out shapes; it holds none of the
method's arithmetic (no slot or block-table computation, no attention, no
quantisation). Both the CUDA path's tests and benchmarks and the CPU oracle
take their inputs from here, and from nowhere else they share.

The workloads stand in for the serving traces the pages measure on (ShareGPT,
Alpaca), which are not used: lengths, head shapes and sharing structure follow
the stated recipes, values are N(0, 1).

A workload is described by
* shapes: ``B`` sequences, ``Hq`` query heads, ``Hkv`` KV heads, ``D`` head dim,
  ``bs`` block size, ``NB`` pool blocks;
* ``free_order``: the initial free list (a seeded permutation of the block ids);
* ``script``: block-manager operations that build the cache state before the
  measured step (``("add", sid)``, ``("append", sid, n)``, ``("fork", p, c)``,
  ``("beam", old_ids, parents, new_ids)``; the random parent draws of a beam
  search are inputs here, each side reshuffles its own manager with them);
* ``step_seqs``: the sequences that append one token in the measured step;
* value tensors, drawn on demand: the past K/V contents of every pool slot
  (``past_pools``), and the step's ``q``, ``k_new``, ``v_new``;
* FP8 scales for the E4M3 variant: ``amax|source| / 448`` per tensor.
"""
import math
from dataclasses import dataclass, field

import numpy as np
import torch

E4M3_MAX = 448.0
_CHUNK_ELEMS = 1 << 26


@dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    bs: int
    NB: int
    seed: int
    scale: float
    src_dtype: torch.dtype            # dtype of q, k_new, v_new and of the pools' source values
    kv_dtype: str                     # "f32", "bf16" or "e4m3"
    free_order: np.ndarray
    script: list
    step_seqs: list
    final_lens: np.ndarray            # length of each sequence after the step (incl. the new token)
    notes: dict = field(default_factory=dict)

    # ---- value tensors --------------------------------------------------
    def _randn(self, shape, tag):
        g = torch.Generator().manual_seed(self.seed * 7919 + tag)
        numel = math.prod(shape)
        out = torch.empty(numel, dtype=self.src_dtype)
        for s in range(0, numel, _CHUNK_ELEMS):
            e = min(numel, s + _CHUNK_ELEMS)
            out[s:e] = torch.randn(e - s, generator=g, dtype=torch.float32).to(self.src_dtype)
        return out.view(*shape)

    def past_pools(self):
        """Source values of every pool slot, ``[NB, Hkv, bs, D]`` in ``src_dtype``.

        For bf16/f32 caches this is the cache content; for the E4M3 cache it is
        what gets quantised into it.
        """
        shape = (self.NB, self.Hkv, self.bs, self.D)
        return self._randn(shape, 1), self._randn(shape, 2)

    def step_inputs(self):
        """``q [B, Hq, D]``, ``k_new [B, Hkv, D]``, ``v_new [B, Hkv, D]`` for the step."""
        q = self._randn((self.B, self.Hq, self.D), 3)
        k = self._randn((self.B, self.Hkv, self.D), 4)
        v = self._randn((self.B, self.Hkv, self.D), 5)
        return q, k, v

    def fp8_scales(self, k_src, v_src, k_new, v_new):
        """Per-tensor scales ``amax|x| / 448`` over the pool sources and new tokens."""
        ks = max(k_src.abs().max().item(), k_new.abs().max().item()) / E4M3_MAX
        vs = max(v_src.abs().max().item(), v_new.abs().max().item()) / E4M3_MAX
        return float(ks), float(vs)

    @property
    def max_blocks_per_seq(self):
        return int(-(-int(self.final_lens.max()) // self.bs))


def _pool_size(total_blocks):
    return int(math.ceil(1.1 * total_blocks))


def prefill_workload(name, seed, lens, Hq, Hkv, D, bs, src_dtype, kv_dtype, scale, NB=None):
    """Sequences 0..B-1, each with ``len - 1`` past tokens and one step token."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int64)
    if NB is None:
        NB = _pool_size(int(sum(-(-int(L) // bs) for L in lens)))
    free_order = rng.permutation(NB)
    script = []
    for b, L in enumerate(lens):
        script.append(("add", b))
        if L > 1:
            script.append(("append", b, int(L) - 1))
    return Workload(name=name, B=len(lens), Hq=Hq, Hkv=Hkv, D=D, bs=bs, NB=NB, seed=seed,
                    scale=scale, src_dtype=src_dtype, kv_dtype=kv_dtype,
                    free_order=free_order, script=script, step_seqs=list(range(len(lens))),
                    final_lens=lens)


def tiny_fp32():
    """4 sequences of lengths {1, 17, 40, 100}, 4 heads (MHA), D 64, bs 16, 64 blocks."""
    return prefill_workload("tiny_fp32", 0, [1, 17, 40, 100], 4, 4, 64, 16,
                             torch.float32, "f32", 1.0 / 8.0, NB=64)


def llama13b_mha_bf16(B=64):
    """LLaMA-13B-shaped layer: 40 heads MHA, D 128, bs 16, lengths U[128, 2048]."""
    rng = np.random.default_rng(1)
    lens = rng.integers(128, 2048, size=B, endpoint=True)
    w = prefill_workload("llama13b_mha_bf16", 1, lens, 40, 40, 128, 16,
                          torch.bfloat16, "bf16", 1.0 / math.sqrt(128))
    return w


def gqa_chat_bf16(B=256):
    """GQA 32 query / 8 KV heads, D 128, bs 16, lengths lognormal(median 400, sigma 1)
    rounded and clipped to [16, 4096]."""
    rng = np.random.default_rng(2)
    lens = np.clip(np.round(400.0 * np.exp(rng.standard_normal(B))), 16, 4096).astype(np.int64)
    return prefill_workload("gqa_chat_bf16", 2, lens, 32, 8, 128, 16,
                             torch.bfloat16, "bf16", 1.0 / math.sqrt(128))


def shared_prefix(fork_step=False, groups=64, per_group=4, prompt=520, max_suffix=256, Hq=40,
                  Hkv=40, D=128, bs=16, kv="bf16", seed=3, name=None):
    """Parallel sampling: ``groups`` prompts of ``prompt`` tokens, each forked into
    ``per_group`` sequences that share the prompt's blocks.

    ``fork_step=True``: every sequence is still at the prompt length, so the step's
    first append into the shared partial block is the copy-on-write step.
    Otherwise each sequence first grows by a suffix ~ U[0, max_suffix] (untimed).
    """
    rng = np.random.default_rng(seed)
    n = groups * per_group
    suffix = np.zeros(n, dtype=np.int64) if fork_step else rng.integers(0, max_suffix, size=n, endpoint=True)
    # pool: every prompt's blocks plus, per sequence, enough blocks for its own tail
    # (the partial prompt block, its suffix and the step token), plus 10%
    per_prompt = -(-prompt // bs)
    own = sum(-(-(prompt % bs + int(s) + 1) // bs) for s in suffix)
    NB = _pool_size(groups * per_prompt + own)
    free_order = rng.permutation(NB)
    script = []
    for g in range(groups):
        parent = g * per_group
        script.append(("add", parent))
        script.append(("append", parent, prompt))
        for c in range(1, per_group):
            script.append(("fork", parent, parent + c))
    if not fork_step:
        for sid in range(n):
            if suffix[sid]:
                script.append(("append", sid, int(suffix[sid])))
    lens = prompt + suffix + 1
    if name is None:
        name = "shared_prefix_fork_bf16" if fork_step else "shared_prefix_bf16"
    src = torch.float32 if kv == "f32" else torch.bfloat16
    return Workload(name=name, B=n, Hq=Hq, Hkv=Hkv, D=D, bs=bs, NB=NB, seed=seed,
                    scale=1.0 / math.sqrt(D), src_dtype=src, kv_dtype=kv,
                    free_order=free_order, script=script, step_seqs=list(range(n)),
                    final_lens=lens, notes={"groups": groups, "per_group": per_group,
                                            "prompt": prompt})


def shared_prefix_bf16(fork_step=False, groups=64, per_group=4, prompt=520, max_suffix=256):
    """64 groups x 4 samples of a 520-token prompt, 40 heads MHA, D 128, bs 16."""
    return shared_prefix(fork_step, groups, per_group, prompt, max_suffix)


def long_fp8(bs=16, B=16, L=32768):
    """Long context with an E4M3 cache: B sequences of L tokens, GQA 32/8, D 128."""
    return prefill_workload(f"long_fp8_bs{bs}", 4, [L] * B, 32, 8, 128, bs,
                             torch.bfloat16, "e4m3", 1.0 / math.sqrt(128))


@dataclass
class ChunkWorkload(Workload):
    """A chunked-prefill step: sequence b appends ``chunks[b]`` tokens at once
    (its chunk) on top of the context the script built, and every chunk token
    is a query."""
    chunks: np.ndarray = None

    @property
    def T(self):
        return int(np.sum(self.chunks))

    @property
    def max_query_len(self):
        return int(np.max(self.chunks)) if len(self.chunks) else 0

    @property
    def query_start(self):
        """Offsets of each sequence's chunk rows in q / out (int32 [B + 1])."""
        return np.concatenate([[0], np.cumsum(self.chunks)]).astype(np.int32)

    def step_inputs(self):
        """``q [T, Hq, D]``, ``k_new [T, Hkv, D]``, ``v_new [T, Hkv, D]``: the chunk
        tokens of sequence 0, then of sequence 1, ..."""
        q = self._randn((self.T, self.Hq, self.D), 3)
        k = self._randn((self.T, self.Hkv, self.D), 4)
        v = self._randn((self.T, self.Hkv, self.D), 5)
        return q, k, v


def chunked_prefill(name, seed, context, chunks, Hq, Hkv, D, bs, NB=None):
    """Sequences 0..B-1 with ``context[b]`` cached tokens, then a chunk of
    ``chunks[b]`` new tokens each (bf16, N(0, 1) values, scale 1/sqrt(D))."""
    rng = np.random.default_rng(seed)
    context = np.asarray(context, dtype=np.int64)
    chunks = np.asarray(chunks, dtype=np.int64)
    lens = context + chunks
    if NB is None:
        NB = _pool_size(int(sum(-(-int(L) // bs) for L in lens)))
    free_order = rng.permutation(NB)
    script = []
    for b, c in enumerate(context):
        script.append(("add", b))
        if c > 0:
            script.append(("append", b, int(c)))
    return ChunkWorkload(name=name, B=len(lens), Hq=Hq, Hkv=Hkv, D=D, bs=bs, NB=NB, seed=seed,
                         scale=1.0 / math.sqrt(D), src_dtype=torch.bfloat16, kv_dtype="bf16",
                         free_order=free_order, script=script, step_seqs=list(range(len(lens))),
                         final_lens=lens, chunks=chunks)


def prefill_llama13b_bf16(B=16, chunk=512):
    """LLaMA-13B-shaped chunked prefill: 40 heads MHA, D 128, bs 16; B sequences
    with a context of U[0, 1536] cached tokens each take a chunk of 512 tokens."""
    rng = np.random.default_rng(5)
    ctx = rng.integers(0, 1536, size=B, endpoint=True)
    return chunked_prefill("prefill_llama13b_bf16", 5, ctx, [chunk] * B, 40, 40, 128, 16)


def prefill_gqa_bf16(B=16, chunk=512):
    """GQA 32 query / 8 KV heads, D 128, bs 16; contexts U[0, 3584], chunks of 512."""
    rng = np.random.default_rng(6)
    ctx = rng.integers(0, 3584, size=B, endpoint=True)
    return chunked_prefill("prefill_gqa_bf16", 6, ctx, [chunk] * B, 32, 8, 128, 16)


@dataclass
class PromptWorkload:
    """Requests given as token ids, for prefix caching: the ``warm`` prompts are
    served first (and released), then every request of ``prompts`` arrives in
    one batch. q/k/v values are N(0, 1), drawn per (phase, request) for a range
    of positions; the pool's earlier content is drawn like the other workloads'.
    """
    name: str
    Hq: int
    Hkv: int
    D: int
    bs: int
    NB: int
    seed: int
    scale: float
    free_order: np.ndarray
    prompts: list
    warm: list
    src_dtype: torch.dtype = torch.bfloat16
    kv_dtype: str = "bf16"

    @property
    def B(self):
        return len(self.prompts)

    @property
    def final_lens(self):
        return np.array([len(p) for p in self.prompts], dtype=np.int64)

    @property
    def max_blocks_per_seq(self):
        return int(-(-int(self.final_lens.max()) // self.bs))

    def _randn(self, shape, tag):
        g = torch.Generator().manual_seed(self.seed * 7919 + tag)
        return torch.randn(*shape, generator=g, dtype=torch.float32).to(self.src_dtype)

    def past_pools(self):
        shape = (self.NB, self.Hkv, self.bs, self.D)
        return self._randn(shape, 1), self._randn(shape, 2)

    def rows(self, phase, b, start, stop):
        """q ``[n, Hq, D]``, k and v ``[n, Hkv, D]`` for positions start..stop-1
        of request b of ``phase`` ("warm" or "step")."""
        n = stop - start
        tag = 1000 + 3 * (b + (0 if phase == "warm" else 100000))
        q = self._randn((n, self.Hq, self.D), tag)
        k = self._randn((n, self.Hkv, self.D), tag + 1)
        v = self._randn((n, self.Hkv, self.D), tag + 2)
        return q, k, v


def system_prompt(B=64, system=1024, suffix=256, Hq=40, Hkv=40, D=128, bs=16, seed=7,
                  vocab=32000, name="prefill_system_prompt_bf16", suffix_lens=None):
    """B requests that all begin with one ``system``-token prompt followed by their
    own ``suffix`` tokens (or ``suffix_lens[b]``); the system prompt alone is
    served first. Token ids uniform in [0, vocab)."""
    rng = np.random.default_rng(seed)
    sys_ids = rng.integers(0, vocab, size=system)
    sl = [suffix] * B if suffix_lens is None else list(suffix_lens)
    prompts = [np.concatenate([sys_ids, rng.integers(0, vocab, size=int(n))]) for n in sl]
    total = -(-system // bs) + sum(-(-(system + int(n)) // bs) for n in sl)
    NB = _pool_size(total)
    return PromptWorkload(name=name, Hq=Hq, Hkv=Hkv, D=D, bs=bs, NB=NB, seed=seed,
                          scale=1.0 / math.sqrt(D), free_order=rng.permutation(NB),
                          prompts=prompts, warm=[sys_ids.copy()])


def beam_search(name, requests, width, prompt, generated, Hq, Hkv, D, bs, seed,
                src_dtype=torch.bfloat16, kv_dtype="bf16"):
    """Beam search: ``requests`` prompts (lengths U[prompt[0], prompt[1]]) with
    ``width`` beams each, after ``generated`` beam steps. Every step each new
    beam's parent is drawn uniformly from its request's old beams (the scores
    that pick them in a real search come from the model), then every beam
    appends its token. The script ends with the measured step's reshuffle; the
    measured step appends one token to each of its beams."""
    rng = np.random.default_rng(seed)
    P = rng.integers(prompt[0], prompt[1], size=requests, endpoint=True)
    script, beams, sid = [], [], 0
    for r in range(requests):
        script += [("add", sid), ("append", sid, int(P[r]))]
        beams.append((sid,))
        sid += 1
    for g in range(generated + 1):
        # one reshuffle of every request's beams: parents index the old beams of
        # all requests, listed request after request
        old, parents, new = [], [], []
        for r in range(requests):
            parents += [len(old) + int(x) for x in rng.integers(0, len(beams[r]), size=width)]
            old += beams[r]
            beams[r] = tuple(range(sid, sid + width))
            new += beams[r]
            sid += width
        script.append(("beam", tuple(old), tuple(parents), tuple(new)))
        if g < generated:
            script += [("append", s, 1) for b in beams for s in b]
    lens = np.repeat(P + generated + 1, width).astype(np.int64)
    NB = _pool_size(int(sum(-(-int(L) // bs) for L in lens)))
    return Workload(name=name, B=requests * width, Hq=Hq, Hkv=Hkv, D=D, bs=bs, NB=NB, seed=seed,
                    scale=1.0 / math.sqrt(D), src_dtype=src_dtype, kv_dtype=kv_dtype,
                    free_order=rng.permutation(NB), script=script,
                    step_seqs=[s for b in beams for s in b], final_lens=lens,
                    notes={"requests": requests, "width": width, "generated": generated,
                           "prompt_lens": P})


def beam_search_bf16(requests=16, width=4, generated=128):
    """LLaMA-13B-shaped beam search: 16 requests x 4 beams (64 sequences), prompts
    U[128, 2048] (the decode batch's length distribution), 128 generated tokens,
    40/40 heads, D 128, bs 16, seed 8."""
    return beam_search("beam_search_bf16", requests, width, (128, 2048), generated, 40, 40, 128,
                       16, 8)


@dataclass
class SwapWorkload:
    """Preemption by swapping: of the decode batch ``base`` (each sequence holding
    its past tokens), the ``victims`` -- the newest arrivals -- are swapped out to
    a host pool of ``num_host_blocks`` blocks and swapped back in, step after step."""
    name: str
    base: Workload
    victims: list
    num_host_blocks: int

    @property
    def victim_blocks(self):
        return int(sum(-(-(int(self.base.final_lens[s]) - 1) // self.base.bs)
                       for s in self.victims))


def swap_llama13b_bf16(B=64, victims=16):
    """The LLaMA-13B-shaped bf16 decode batch (B sequences, lengths U[128, 2048]);
    its last ``victims`` sequences are preempted by swapping."""
    base = llama13b_mha_bf16(B)
    v = list(range(B - min(victims, B), B))
    sw = SwapWorkload("swap_llama13b_bf16", base, v, 0)
    sw.num_host_blocks = _pool_size(sw.victim_blocks)
    return sw


SWAP_CONFIGS = {
    "swap_llama13b_bf16": swap_llama13b_bf16,
}


PREFILL_CONFIGS = {
    "prefill_llama13b_bf16": prefill_llama13b_bf16,
    "prefill_gqa_bf16": prefill_gqa_bf16,
}

# prefix caching: 64 requests sharing a 1024-token system prompt (LLaMA-13B shape)
PROMPT_CONFIGS = {
    "prefill_system_prompt_bf16": system_prompt,
}


CONFIGS = {
    "tiny_fp32": tiny_fp32,
    "llama13b_mha_bf16": llama13b_mha_bf16,
    "gqa_chat_bf16": gqa_chat_bf16,
    "shared_prefix_bf16": shared_prefix_bf16,
    "shared_prefix_fork_bf16": lambda: shared_prefix_bf16(fork_step=True),
    "long_fp8_bs16": lambda: long_fp8(16),
    "long_fp8_bs32": lambda: long_fp8(32),
    "beam_search_bf16": beam_search_bf16,
}
