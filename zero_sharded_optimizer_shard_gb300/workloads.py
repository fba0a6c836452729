"""Parameter lists and synthetic-input recipes of the ZeRO-3 workloads.

Pure data: tensor shapes, submodule membership, AdamW hyper-parameters and
the generator settings of each workload.  Nothing here computes any part of
the sharded optimizer step; the same lists feed the CPU oracle, the CUDA
library, the tests and the benchmark.

Hyper-parameters follow the AdamW block of the example DeepSpeed config in
the ZERO tutorial (cnhsyj.com/news/20093, section 3.1 "基礎配置與啟動"):
lr 5e-5, betas (0.9, 0.999), eps 1e-8, weight_decay 0.01, held constant.
The persistence threshold 1e5 and the reduce and all-gather bucket sizes
5e8 are the defaults quoted in
"DeepSpeed Zero-3 的参数分区与按需访问机制" (hotelren.com/news/4329759) and in
its minimal ZeRO-3 config.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

PERSISTENCE_THRESHOLD = 100_000
REDUCE_BUCKET_SIZE = 500_000_000
# parameter gathers are grouped into buckets of this many elements
# (allgather_bucket_size of the same minimal config)
ALLGATHER_BUCKET_SIZE = 500_000_000

ADAMW = dict(lr=5e-5, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)

# generator stream ids (keys of the counter-based generator)
STREAM_MASTER = 1          # fp32 master init of the partitioned flat buffer
STREAM_MASTER_PERSIST = 2  # fp32 master init of the persistent group
STREAM_GRAD = 3            # bf16 local gradients, partitioned flat index
STREAM_GRAD_PERSIST = 4    # bf16 local gradients, persistent index
STREAM_RAGGED_SIZES = 5    # tensor sizes of the ragged list
STREAM_RAGGED_GROUPS = 6   # submodule run lengths of the ragged list


@dataclass
class Workload:
    name: str
    numels: List[int]
    submodule_of: List[int]
    n_ranks: int
    steps: int
    seed: int
    master_sigma: float = 0.02
    grad_sigma: float = 1e-3
    outlier_p: float = 0.0
    outlier_sigma: float = 1e-1
    threshold: int = PERSISTENCE_THRESHOLD
    bucket: int = REDUCE_BUCKET_SIZE
    gather_bucket: int = ALLGATHER_BUCKET_SIZE
    hparams: dict = field(default_factory=lambda: dict(ADAMW))
    names: Optional[List[str]] = None
    # rank-0 view: only ranks in `ranks` hold optimizer state on this device
    ranks: Optional[List[int]] = None

    @property
    def psi(self) -> int:
        return sum(self.numels)


def _add(names, numels, subs, name, numel, sub):
    names.append(name)
    numels.append(int(numel))
    subs.append(int(sub))


def toy_mlp() -> Workload:
    """2-layer MLP 784-1024-256-10 with biases; N_d=2, 3 steps, seed 1."""
    names, numels, subs = [], [], []
    dims = [(784, 1024), (1024, 256), (256, 10)]
    for k, (i, o) in enumerate(dims):
        _add(names, numels, subs, f"fc{k}.weight", i * o, k)
        _add(names, numels, subs, f"fc{k}.bias", o, k)
    return Workload("toy_mlp", numels, subs, n_ranks=2, steps=3, seed=1, names=names)


def gpt2_like(n_layer: int, d: int, vocab: int, n_ctx: int) -> tuple:
    """GPT-2 style decoder parameter list in named_parameters order.

    Tied LM head (no extra tensor), LayerNorm weight+bias, Conv1D biases.
    Submodules: 0 = token+position embeddings, 1..n_layer = blocks,
    n_layer+1 = final LayerNorm.
    """
    names, numels, subs = [], [], []
    _add(names, numels, subs, "wte", vocab * d, 0)
    _add(names, numels, subs, "wpe", n_ctx * d, 0)
    for l in range(n_layer):
        s = l + 1
        p = f"h.{l}."
        _add(names, numels, subs, p + "ln_1.weight", d, s)
        _add(names, numels, subs, p + "ln_1.bias", d, s)
        _add(names, numels, subs, p + "attn.c_attn.weight", d * 3 * d, s)
        _add(names, numels, subs, p + "attn.c_attn.bias", 3 * d, s)
        _add(names, numels, subs, p + "attn.c_proj.weight", d * d, s)
        _add(names, numels, subs, p + "attn.c_proj.bias", d, s)
        _add(names, numels, subs, p + "ln_2.weight", d, s)
        _add(names, numels, subs, p + "ln_2.bias", d, s)
        _add(names, numels, subs, p + "mlp.c_fc.weight", d * 4 * d, s)
        _add(names, numels, subs, p + "mlp.c_fc.bias", 4 * d, s)
        _add(names, numels, subs, p + "mlp.c_proj.weight", 4 * d * d, s)
        _add(names, numels, subs, p + "mlp.c_proj.bias", d, s)
    _add(names, numels, subs, "ln_f.weight", d, n_layer + 1)
    _add(names, numels, subs, "ln_f.bias", d, n_layer + 1)
    return names, numels, subs


def gpt2_small() -> Workload:
    """GPT-2-small shaped list (~124M); N_d=4; 1% outlier gradients; 10 steps."""
    names, numels, subs = gpt2_like(12, 768, 50257, 1024)
    return Workload("gpt2_small", numels, subs, n_ranks=4, steps=10, seed=2,
                    outlier_p=0.01, names=names)


def decoder_1p3b() -> Workload:
    """1.3B GPT-style decoder (24 layers, d=2048, vocab 50257, n_ctx 2048); N_d=8."""
    names, numels, subs = gpt2_like(24, 2048, 50257, 2048)
    return Workload("decoder_1p3b", numels, subs, n_ranks=8, steps=20, seed=4, names=names)


def llama_7b(rank0_view: bool = True) -> Workload:
    """Llama-7B shaped list (32 layers, d=4096, SwiGLU 11008, vocab 32000,
    RMSNorm, untied head) in HF named_parameters order; N_d=8.

    Submodules: 0 = embed_tokens, 1..32 = decoder layers, 33 = final norm,
    34 = lm_head.
    """
    d, f, vocab, L = 4096, 11008, 32000, 32
    names, numels, subs = [], [], []
    _add(names, numels, subs, "embed_tokens.weight", vocab * d, 0)
    for l in range(L):
        s = l + 1
        p = f"layers.{l}."
        for proj in ("q_proj", "k_proj", "v_proj", "o_proj"):
            _add(names, numels, subs, p + f"self_attn.{proj}.weight", d * d, s)
        _add(names, numels, subs, p + "mlp.gate_proj.weight", f * d, s)
        _add(names, numels, subs, p + "mlp.up_proj.weight", f * d, s)
        _add(names, numels, subs, p + "mlp.down_proj.weight", d * f, s)
        _add(names, numels, subs, p + "input_layernorm.weight", d, s)
        _add(names, numels, subs, p + "post_attention_layernorm.weight", d, s)
    _add(names, numels, subs, "norm.weight", d, L + 1)
    _add(names, numels, subs, "lm_head.weight", vocab * d, L + 2)
    return Workload("llama_7b_rank0" if rank0_view else "llama_7b", numels, subs,
                    n_ranks=8, steps=10, seed=5, names=names,
                    ranks=[0] if rank0_view else None)


def ragged(n_tensors: int = 2000, n_ranks: int = 7, seed: int = 3,
           small_hi: float = 1e5, big_lo: float = 1e5, big_hi: float = 4e6,
           p_small: float = 0.30, steps: int = 5) -> Workload:
    """Ragged-shape stress list.

    Sizes are a p_small / (1 - p_small) mixture of log-uniform [1, small_hi)
    and log-uniform [big_lo, big_hi], redrawn while divisible by n_ranks
    (for n_ranks > 1; at most 64 draws per tensor, the last one kept).
    Submodules are consecutive runs of 1..8 tensors.  All draws come from the
    counter-based generator (see synth.uniform_u64), so the list is a pure
    function of the seed.
    """
    from . import synth  # local import: synth has no dependency back here

    numels = []
    draw = 0
    for t in range(n_tensors):
        while True:
            u = synth.uniform_u64(seed, STREAM_RAGGED_SIZES, 0, 0, [t * 64 + draw])[0]
            draw += 1
            pick = (int(u) >> 40) / float(1 << 24)          # component choice
            frac = (int(u) & ((1 << 40) - 1)) / float(1 << 40)  # position in log range
            if pick < p_small:
                lo, hi = 1.0, small_hi
            else:
                lo, hi = big_lo, big_hi
            size = int(math.floor(math.exp(math.log(lo) + frac * (math.log(hi) - math.log(lo)))))
            top = int(hi) - 1 if pick < p_small else int(hi)
            size = min(max(size, int(lo)), top)
            if n_ranks <= 1 or size % n_ranks != 0 or draw == 64:
                break
        draw = 0
        numels.append(size)
    subs = []
    k = 0
    t = 0
    while t < n_tensors:
        u = synth.uniform_u64(seed, STREAM_RAGGED_GROUPS, 0, 0, [k])[0]
        run = 1 + int(u >> 61)  # 1..8
        for _ in range(min(run, n_tensors - t)):
            subs.append(k)
            t += 1
        k += 1
    names = [f"t{t}" for t in range(n_tensors)]
    return Workload(f"ragged_{n_tensors}", numels, subs, n_ranks=n_ranks, steps=steps,
                    seed=seed, names=names)


def ragged_small(n_ranks: int = 7) -> Workload:
    """The ragged recipe scaled down so the whole oracle runs in seconds:
    300 tensors, persistence threshold 1e3, sizes a 30/70 mixture of
    log-uniform [1, 1e3) and [1e3, 4e4]."""
    w = ragged(n_tensors=300, n_ranks=n_ranks, small_hi=1e3, big_lo=1e3, big_hi=4e4)
    w.threshold = 1000
    w.name = f"ragged_small_nd{n_ranks}"
    return w


def mini_gpt(n_ranks: int = 4) -> Workload:
    """Two-block GPT with d=256: many kernel tiles and a ragged tail, small
    enough for the full oracle."""
    names, numels, subs = gpt2_like(2, 256, 1000, 128)
    return Workload(f"mini_gpt_nd{n_ranks}", numels, subs, n_ranks=n_ranks, steps=10,
                    seed=7, outlier_p=0.01, names=names)


BY_NAME = {
    "toy_mlp": toy_mlp,
    "gpt2_small": gpt2_small,
    "ragged": ragged,
    "decoder_1p3b": decoder_1p3b,
    "llama_7b_rank0": llama_7b,
}
