"""Seeded synthetic inputs shared by the CUDA path and the CPU oracle.

This module only draws random numbers and describes model shapes.  It holds
none of the forward's arithmetic: no normalisation, no quantisation rule, no
reduction.  Where a tensor has to be handed over in bf16 or e4m3, the
narrowing is done by PyTorch's own dtype cast (a library routine), so that
neither side supplies the other's inputs.

The workloads mirror the ones the pages describe:

* "No More Train-Inference Mismatch: Bitwise Consistent On-Policy
  Reinforcement Learning with vLLM and TorchTitan", section "实验环境"
  (experimental setup): a Qwen3-1.7B policy, GSM8K prompts;
* "Finish RL Training Faster: Bitwise-Consistent, High-Performance,
  Agent-Driven", section "两组结果，要连同分母一起读" (results): FP8 KV cache,
  MoE with top-k routing, sparse attention, and a Mamba-2 hybrid.

The pages' datasets (GSM8K, DAPO maths, SWE-bench Pro) are not used: token
ids are uniform random integers with the lengths stated below.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Dict, List

import numpy as np
import torch


# --------------------------------------------------------------------------
# model shapes
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class DenseConfig:
    """A pre-norm decoder with GQA attention and a SiLU-gated MLP."""

    name: str
    layers: int
    hidden: int
    q_heads: int
    kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    rope_theta: float
    eps: float
    qk_norm: bool
    tied: bool
    kv_fp8: bool = False
    page: int = 64           # tokens per KV page
    kv_split: int = 1024     # tokens per attention KV split (model constant)

    @property
    def qkv_width(self) -> int:
        return (self.q_heads + 2 * self.kv_heads) * self.head_dim


TINY = DenseConfig(
    name="tiny-dense-2L-h256", layers=2, hidden=256, q_heads=4, kv_heads=2,
    head_dim=64, intermediate=688, vocab=4096, rope_theta=1e6, eps=1e-6,
    qk_norm=False, tied=False)

QWEN3_1P7B = DenseConfig(
    name="qwen3-1.7b-shape", layers=28, hidden=2048, q_heads=16, kv_heads=8,
    head_dim=128, intermediate=6144, vocab=151936, rope_theta=1e6, eps=1e-6,
    qk_norm=True, tied=True)

QWEN3_1P7B_FP8KV = replace(QWEN3_1P7B, name="qwen3-1.7b-shape-fp8kv", kv_fp8=True)


def scaled_dense(cfg: DenseConfig, layers: int) -> DenseConfig:
    """Same per-layer shape with fewer layers (for oracle-sized parity cases)."""
    return replace(cfg, name=f"{cfg.name}-{layers}L", layers=layers)


@dataclass(frozen=True)
class MoEConfig:
    """One MoE + sparse-attention block (routed experts in FP8, 128x128 scales)."""

    hidden: int = 4096
    experts: int = 64
    top_k: int = 6
    expert_inter: int = 1408
    tokens: int = 4096
    context: int = 32768
    index_topk: int = 2048
    index_dim: int = 128
    attn_heads: int = 32
    attn_kv_heads: int = 1
    head_dim: int = 128


MOE_BLOCK = MoEConfig()


@dataclass(frozen=True)
class SSDConfig:
    """Mamba-2 SSD mixer shape (one B/C group)."""

    d_model: int = 2560
    heads: int = 64
    head_dim: int = 64
    state: int = 128
    chunk: int = 256


SSD_LAYER = SSDConfig()


# --------------------------------------------------------------------------
# random sources
# --------------------------------------------------------------------------
def rng(seed: int) -> np.random.Generator:
    """Counter-based generator (Philox) so streams are reproducible on any host."""
    return np.random.Generator(np.random.Philox(seed))


def normal_f32(g: np.random.Generator, shape, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    return (g.standard_normal(size=shape, dtype=np.float32) * np.float32(std)
            + np.float32(mean)).astype(np.float32)


def to_bf16(x: np.ndarray) -> torch.Tensor:
    """Narrow fp32 data to a bf16 CPU tensor with PyTorch's cast."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw uint16 payload of a bf16 tensor (for the oracle's own decoder)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def fp8_bits(t: torch.Tensor) -> np.ndarray:
    """Raw uint8 payload of a float8_e4m3fn tensor."""
    return t.contiguous().view(torch.uint8).numpy().copy()


def normal_bf16(g: np.random.Generator, shape, std: float = 1.0) -> torch.Tensor:
    return to_bf16(normal_f32(g, shape, std))


# --------------------------------------------------------------------------
# dense decoder weights
# --------------------------------------------------------------------------
def dense_weights(cfg: DenseConfig, seed: int = 0, std: float = 0.02,
                  random_gains: bool = False, lm_scale: float = 1.0) -> Dict[str, torch.Tensor]:
    """Random-init bf16 weights of the decoder, N(0, std) from a seed.

    Norm gains are 1.0 (fresh init) unless ``random_gains``; ``lm_scale``
    multiplies the LM-head draw (a "peaked" variant whose logits are far from
    uniform, so that log-softmax is exercised beyond -log V).
    """
    g = rng(seed)
    d, D, I = cfg.hidden, cfg.head_dim, cfg.intermediate
    W: Dict[str, torch.Tensor] = {}
    W["embed"] = normal_bf16(g, (cfg.vocab, d), std)

    def gain(n):
        if random_gains:
            return to_bf16(1.0 + normal_f32(g, (n,), 0.1))
        return to_bf16(np.ones(n, np.float32))

    for l in range(cfg.layers):
        p = f"l{l}."
        W[p + "attn_norm"] = gain(d)
        W[p + "wqkv"] = normal_bf16(g, (cfg.qkv_width, d), std)
        if cfg.qk_norm:
            W[p + "q_norm"] = gain(D)
            W[p + "k_norm"] = gain(D)
        W[p + "wo"] = normal_bf16(g, (d, cfg.q_heads * D), std)
        W[p + "mlp_norm"] = gain(d)
        W[p + "wgu"] = normal_bf16(g, (2 * I, d), std)       # rows [gate | up]
        W[p + "wd"] = normal_bf16(g, (d, I), std)
    W["final_norm"] = gain(d)
    if cfg.tied and lm_scale == 1.0:
        W["lm_head"] = W["embed"]
    else:
        src = W["embed"].float().numpy() if cfg.tied else normal_f32(g, (cfg.vocab, d), std)
        W["lm_head"] = to_bf16(src * np.float32(lm_scale))
    return W


# --------------------------------------------------------------------------
# token workloads
# --------------------------------------------------------------------------
@dataclass
class Sequence:
    tokens: np.ndarray        # int32 [prompt_len + response_len]
    prompt_len: int

    @property
    def length(self) -> int:
        return int(self.tokens.shape[0])


def tiny_sequences(cfg: DenseConfig, n: int = 8, lo: int = 16, hi: int = 128,
                   seed: int = 1) -> List[Sequence]:
    """n sequences, lengths uniform in [lo, hi], ids uniform over the vocabulary.

    The prompt is the first quarter of each sequence (at least one token).
    """
    g = rng(seed)
    out = []
    for _ in range(n):
        L = int(g.integers(lo, hi + 1))
        toks = g.integers(0, cfg.vocab, size=L, dtype=np.int64).astype(np.int32)
        out.append(Sequence(toks, max(1, L // 4)))
    return out


def rollout_sequences(cfg: DenseConfig, prompts: int = 64, responses: int = 8,
                      prompt_lo: int = 64, prompt_hi: int = 512,
                      resp_lo: int = 128, resp_hi: int = 1024, seed: int = 1) -> List[Sequence]:
    """GRPO-shaped batch: each prompt is shared by ``responses`` sampled answers.

    Response ids are drawn in advance (teacher forcing): the sampler is not part
    of the logprob path, so the rollout consumes pre-drawn tokens.
    """
    g = rng(seed)
    out = []
    for _ in range(prompts):
        P = int(g.integers(prompt_lo, prompt_hi + 1))
        prompt = g.integers(0, cfg.vocab, size=P, dtype=np.int64).astype(np.int32)
        for _ in range(responses):
            R = int(g.integers(resp_lo, resp_hi + 1))
            resp = g.integers(0, cfg.vocab, size=R, dtype=np.int64).astype(np.int32)
            out.append(Sequence(np.concatenate([prompt, resp]), P))
    return out


# --------------------------------------------------------------------------
# per-op inputs
# --------------------------------------------------------------------------
def e4m3_from_f32(x: np.ndarray) -> torch.Tensor:
    """Narrow fp32 data (already inside +-448) to float8_e4m3fn with PyTorch's cast."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)


def fp8_block_weights(g: np.random.Generator, groups: int, n: int, k: int):
    """Expert weights as e4m3 codes with one fp32 scale per 128x128 block.

    Codes come from N(0, 64) clipped to the finite range; scales are drawn
    log-uniformly so that code*scale has magnitude near 0.02.
    """
    codes = e4m3_from_f32(np.clip(normal_f32(g, (groups, n, k), 64.0), -448, 448))
    nb, kb = (n + 127) // 128, (k + 127) // 128
    scales = (np.float32(0.02 / 64.0)
              * np.exp2(g.uniform(-1.0, 1.0, size=(groups, nb, kb))).astype(np.float32))
    return codes, scales.astype(np.float32)


def ssd_inputs(g: np.random.Generator, T: int, cfg: SSDConfig = SSD_LAYER):
    """Mamba-2 SSD inputs: x, B, C ~ N(0,1) (bf16), dt = softplus(N(-3,1)) (fp32),
    A = -U[1,16] per head, D ~ N(0,1) per head."""
    H, P, N = cfg.heads, cfg.head_dim, cfg.state
    x = normal_bf16(g, (T, H, P))
    B = normal_bf16(g, (T, N))
    C = normal_bf16(g, (T, N))
    dt = np.log1p(np.exp(normal_f32(g, (T, H), 1.0, -3.0))).astype(np.float32)
    A = (-g.uniform(1.0, 16.0, size=H)).astype(np.float32)
    D = normal_f32(g, (H,))
    return x, dt, A, B, C, D
