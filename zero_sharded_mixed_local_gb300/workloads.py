"""Workload shapes and seeded synthetic inputs for the ZeRO-1 local-shard step.

This module only describes parameter lists and draws random numbers.  It
holds none of the method's arithmetic (no sharding, no accumulation, no
norm, no optimizer math): callers give it the per-tensor shard sizes and the
arena offsets, and it fills buffers with seeded values.  Both the CUDA path
and the CPU oracle are fed from the same draw.

Parameter lists follow the Llama/SmolLM layout the "Nanotron Guide" trains
(section "YAML configuration": SmolLM-1.7B with 24 layers, hidden 2048,
vocab 49152, tied embeddings) with RMSNorm weights as the tensors excluded
from weight decay.  Order is the usual module order: embedding, then per
layer q, k, v, o, gate, up, down, input norm, post-attention norm, then the
final norm and (when untied) the output head.
"""
from dataclasses import dataclass, field
from typing import List, Optional

import math

import numpy as np
import torch


@dataclass
class ParamList:
    names: List[str]
    numels: List[int]
    no_decay: List[int]

    @property
    def total(self) -> int:
        return int(sum(self.numels))

    def __len__(self):
        return len(self.numels)


def llama_style(vocab, hidden, ffn, layers, n_heads, n_kv_heads, head_dim, tied) -> ParamList:
    names, numels, nd = [], [], []

    def add(name, n, no_decay=0):
        names.append(name)
        numels.append(int(n))
        nd.append(no_decay)

    add("embed_tokens.weight", vocab * hidden)
    q_out, kv_out = n_heads * head_dim, n_kv_heads * head_dim
    for i in range(layers):
        p = "layers.%d." % i
        add(p + "self_attn.q_proj.weight", q_out * hidden)
        add(p + "self_attn.k_proj.weight", kv_out * hidden)
        add(p + "self_attn.v_proj.weight", kv_out * hidden)
        add(p + "self_attn.o_proj.weight", hidden * q_out)
        add(p + "mlp.gate_proj.weight", ffn * hidden)
        add(p + "mlp.up_proj.weight", ffn * hidden)
        add(p + "mlp.down_proj.weight", hidden * ffn)
        add(p + "input_layernorm.weight", hidden, 1)
        add(p + "post_attention_layernorm.weight", hidden, 1)
    add("norm.weight", hidden, 1)
    if not tied:
        add("lm_head.weight", vocab * hidden)
    return ParamList(names, numels, nd)


def ragged_list(n_tensors=20000, max_log2=22, no_decay_frac=0.1, seed=0) -> ParamList:
    """Sizes floor(exp(U(0, max_log2 * ln 2))), i.e. log-uniform in [1, 2^max_log2)."""
    rng = np.random.default_rng(seed)
    u = rng.uniform(0.0, max_log2 * math.log(2.0), n_tensors)
    sizes = np.clip(np.floor(np.exp(u)).astype(np.int64), 1, 1 << max_log2)
    nd = (rng.random(n_tensors) < no_decay_frac).astype(int)
    return ParamList(["t%05d" % i for i in range(n_tensors)], [int(s) for s in sizes], [int(x) for x in nd])


@dataclass
class Workload:
    name: str
    description: str
    params: ParamList
    dp_size: int
    dp_rank: int
    micro_batches: int            # K
    steps: int
    grad_sigma: float             # std of each micro-batch gradient element
    per_tensor_scale: Optional[tuple] = None   # (lo, hi): per-tensor log-uniform grad scale
    target_norm: Optional[float] = None        # set sigma so the accumulated local norm is ~this
    hp: dict = field(default_factory=lambda: dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8,
                                                  weight_decay=0.1, clip_grad=1.0))
    seed: int = 0
    # optional parameter groups (0..7) with per-group lr / weight-decay multipliers
    groups: Optional[list] = None
    lr_scale: Optional[list] = None
    wd_scale: Optional[list] = None

    def plan_kwargs(self):
        if self.groups is None:
            return {"no_decay": self.params.no_decay}
        return {"groups": self.groups, "lr_scale": self.lr_scale, "wd_scale": self.wd_scale}

    def group_scales(self):
        """(lr_scale[8], wd_scale[8]) the step applies per group."""
        if self.groups is None:
            return [1.0] * 8, [1.0, 0.0] + [1.0] * 6
        return list(self.lr_scale or [1.0] * 8), list(self.wd_scale or [1.0, 0.0] + [1.0] * 6)


def _toy():
    return llama_style(4096, 256, 1024, 2, 4, 4, 64, tied=True)


def _smollm135m():
    return llama_style(49152, 576, 1536, 30, 9, 3, 64, tied=True)


def _smollm1p7b():
    return llama_style(49152, 2048, 8192, 24, 32, 32, 64, tied=True)


def _llama8b():
    return llama_style(128256, 4096, 14336, 32, 32, 8, 128, tied=False)


def get_workload(name: str) -> Workload:
    if name == "toy":
        return Workload("toy", "toy Llama-style list (vocab 4096, hidden 256, ffn 1024, 2 layers), "
                        "dp4 rank0, K=2", _toy(), 4, 0, 2, 3, 1e-3)
    if name == "smollm135m":
        return Workload("smollm135m", "SmolLM-135M-shaped list, dp1 (full list), K=4, per-tensor "
                        "grad scale log-uniform [0.1, 10]", _smollm135m(), 1, 0, 4, 10, 1e-3,
                        per_tensor_scale=(0.1, 10.0))
    if name == "smollm1p7b":
        return Workload("smollm1p7b", "SmolLM-1.7B-shaped list, dp8 rank3, K=8, accumulated norm ~4",
                        _smollm1p7b(), 8, 3, 8, 10, 1e-3, target_norm=4.0)
    if name == "llama8b":
        return Workload("llama8b", "Llama-3.1-8B-shaped list (untied), dp8 rank0 "
                        "(1,003,782,656 local params), K=1", _llama8b(), 8, 0, 1, 20, 1e-3)
    if name == "smollm135m_mup":
        # hidden matrices in group 0 at lr * 64/576 (a muP transfer from a width-64 proxy),
        # norm weights in group 1 (no decay), embedding in group 2 at the base lr and half decay
        pl = _smollm135m()
        grp = [1 if "norm" in n else (2 if "embed" in n else 0) for n in pl.names]
        return Workload("smollm135m_mup", "SmolLM-135M-shaped list with muP groups (hidden lr x 64/576), dp2 "
                        "rank1, K=2", pl, 2, 1, 2, 5, 1e-3, groups=grp,
                        lr_scale=[64 / 576, 1.0, 1.0] + [1.0] * 5, wd_scale=[1.0, 0.0, 0.5] + [1.0] * 5)
    if name == "ragged":
        return Workload("ragged", "ragged stress list: 20,000 tensors log-uniform in [1, 2^22], 10% "
                        "no-decay, dp2 rank1, K=4", ragged_list(), 2, 1, 4, 5, 1e-2)
    raise KeyError(name)


WORKLOADS = ("toy", "smollm135m", "smollm1p7b", "llama8b", "ragged")


@dataclass
class Layout:
    """Where each tensor's local shard lives: counts and arena offsets (elements)."""
    counts: np.ndarray
    offsets: np.ndarray
    no_decay: np.ndarray
    arena_numel: int

    @staticmethod
    def packed(counts, no_decay):
        counts = np.asarray(counts, np.int64)
        offs = np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(np.int64) if len(counts) else counts
        return Layout(counts, offs, np.asarray(no_decay, np.uint8), int(counts.sum()))


def _grad_sigma(w: Workload, local_numel: int) -> float:
    if w.target_norm is not None and local_numel > 0:
        return w.target_norm / math.sqrt(w.micro_batches * local_numel)
    return w.grad_sigma


class InputGenerator:
    """Seeded draws into arena-shaped tensors (padding stays zero).

    Every quantity is drawn tensor by tensor in plan order from one
    torch.Generator on ``device``, so a given (seed, layout, device) always
    gives the same values.
    """

    def __init__(self, workload: Workload, layout: Layout, device="cpu", seed=None):
        self.w = workload
        self.layout = layout
        self.device = torch.device(device)
        self.seed = workload.seed if seed is None else seed
        self.gen = torch.Generator(device=self.device)
        self.gen.manual_seed(self.seed)
        self.sigma = _grad_sigma(workload, int(layout.counts.sum()))
        if workload.per_tensor_scale is not None:
            lo, hi = workload.per_tensor_scale
            rng = np.random.default_rng(self.seed + 17)
            self.tensor_scale = np.exp(rng.uniform(math.log(lo), math.log(hi), len(layout.counts)))
        else:
            self.tensor_scale = None

    def _segments(self):
        L = self.layout
        for i in range(len(L.counts)):
            c = int(L.counts[i])
            if c:
                yield i, int(L.offsets[i]), c

    def master(self) -> torch.Tensor:
        """fp32 master weights: N(0, 0.02) for decayed tensors, 1.0 for norm weights."""
        out = torch.zeros(self.layout.arena_numel, dtype=torch.float32, device=self.device)
        for i, o, c in self._segments():
            if self.layout.no_decay[i]:
                out[o:o + c].fill_(1.0)
            else:
                out[o:o + c].normal_(0.0, 0.02, generator=self.gen)
        return out

    def zeros(self, dtype=torch.float32) -> torch.Tensor:
        return torch.zeros(self.layout.arena_numel, dtype=dtype, device=self.device)

    def micro_grad(self, out=None) -> torch.Tensor:
        """One bf16 micro-batch gradient: N(0, sigma^2) (times the per-tensor scale), RNE to bf16.
        ``out``: an arena this fills instead of a new one (its padding must be zero; only the
        shards are written)."""
        if out is None:
            out = torch.zeros(self.layout.arena_numel, dtype=torch.bfloat16, device=self.device)
        tmp = None
        for i, o, c in self._segments():
            if tmp is None or tmp.numel() < c:
                tmp = torch.empty(max(c, 1 << 20), dtype=torch.float32, device=self.device)
            t = tmp[:c]
            t.normal_(0.0, self.sigma, generator=self.gen)
            if self.tensor_scale is not None:
                t.mul_(float(self.tensor_scale[i]))
            out[o:o + c].copy_(t)
        return out

    def micro_grads(self, k=None, out=None) -> List[torch.Tensor]:
        """K micro-batch gradients, drawn in order; ``out`` (a list of arenas) is refilled if given."""
        if out is not None:
            return [self.micro_grad(o) for o in out]
        return [self.micro_grad() for _ in range(self.w.micro_batches if k is None else k)]


def gather_shards(arena: torch.Tensor, layout: Layout) -> torch.Tensor:
    """Concatenate the shards of an arena in plan order, dropping padding."""
    pieces = [arena[int(o):int(o) + int(c)] for o, c in zip(layout.offsets, layout.counts) if c]
    if not pieces:
        return arena[:0].clone()
    return torch.cat(pieces)
