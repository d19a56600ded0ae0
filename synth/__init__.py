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


@dataclass(frozen=True)
class HybridConfig:
    """Mamba-2 / attention hybrid: ``pattern`` lists the mixers of the stack
    ("M" Mamba-2, "A" GQA attention), each followed by a SiLU-gated MLP."""

    name: str
    d_model: int
    ssd_heads: int
    ssd_head_dim: int
    state: int
    chunk: int
    q_heads: int
    kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    pattern: str = "MMMMA"
    eps: float = 1e-6
    rope_theta: float = 1e6
    page: int = 64
    kv_split: int = 1024
    kv_fp8: bool = False
    conv_width: int = 4

    @property
    def d_inner(self) -> int:
        return self.ssd_heads * self.ssd_head_dim

    @property
    def conv_channels(self) -> int:
        return self.d_inner + 2 * self.state

    @property
    def in_proj_width(self) -> int:
        return 2 * self.d_inner + 2 * self.state + self.ssd_heads

    @property
    def qkv_width(self) -> int:
        return (self.q_heads + 2 * self.kv_heads) * self.head_dim

    @property
    def layers(self) -> int:          # attention layers (the ones with a KV cache)
        return self.pattern.count("A")


# one hybrid unit at the Nemotron-style width (vocabulary: a reading, the
# pages give none)
HYBRID = HybridConfig(name="mamba2-hybrid-unit-d2560", d_model=2560, ssd_heads=64, ssd_head_dim=64,
                      state=128, chunk=256, q_heads=32, kv_heads=4, head_dim=80, intermediate=6912,
                      vocab=131072)
HYBRID_TINY = HybridConfig(name="mamba2-hybrid-tiny", d_model=256, ssd_heads=8, ssd_head_dim=64,
                           state=128, chunk=256, q_heads=4, kv_heads=2, head_dim=80, intermediate=512,
                           vocab=4096)


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


# --------------------------------------------------------------------------
# device-side draws for throughput workloads (no oracle comparison)
# --------------------------------------------------------------------------
def device_generator(seed: int, device="cuda") -> torch.Generator:
    """torch's counter-based CUDA generator (Philox), seeded."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return gen


def device_normal(gen: torch.Generator, shape, std: float = 1.0, dtype=torch.bfloat16) -> torch.Tensor:
    """N(0, std^2) draws made on the device, narrowed by PyTorch's cast."""
    return (torch.randn(*shape, generator=gen, device=gen.device) * std).to(dtype)


def device_fp8_block_weights(gen: torch.Generator, groups: int, n: int, k: int):
    """The recipe of ``fp8_block_weights`` drawn on the device: e4m3 codes of
    N(0, 64) clipped to the finite range, one log-uniform fp32 scale (around
    0.02 / 64) per 128x128 block.  Returns (codes uint8 [groups, n, k],
    scales fp32 [groups, ceil(n/128), ceil(k/128)])."""
    dev = gen.device
    codes = torch.empty(groups, n, k, dtype=torch.uint8, device=dev)
    for gi in range(groups):   # one group at a time keeps the fp32 draw small
        x = (torch.randn(n, k, generator=gen, device=dev) * 64.0).clamp_(-448, 448)
        codes[gi] = x.to(torch.float8_e4m3fn).view(torch.uint8)
    nb, kb = (n + 127) // 128, (k + 127) // 128
    u = torch.rand(groups, nb, kb, generator=gen, device=dev) * 2.0 - 1.0
    return codes, (0.02 / 64.0) * torch.exp2(u)


# --------------------------------------------------------------------------
# hybrid stack weights (NVFP4 linear layers)
# --------------------------------------------------------------------------
# magnitudes of the 8 non-negative e2m1 codes 0..7 (0, 0.5, 1, 1.5, 2, 3, 4, 6)
# are drawn with these probabilities (a bell-shaped spread over the grid);
# the sign bit (code bit 3) is a fair coin
_E2M1_MAG_P = np.array([0.12, 0.22, 0.20, 0.16, 0.12, 0.10, 0.05, 0.03])


def nvfp4_weights(g: np.random.Generator, n: int, k: int):
    """NVFP4 weights drawn as codes, in the packed storage: e2m1 codes uint8
    [n, k/2] (two per byte, element 2i in the low nibble of byte i) and e4m3
    scale codes uint8 [n, k/16] drawn uniformly from 0x04..0x0F (scales 2^-7 ..
    1.875 * 2^-6, so code x scale has an RMS near 0.03).  No quantisation
    happens here: each side decodes the codes with its own codec.  k is a
    multiple of 16."""
    mag = g.choice(8, size=(n, k), p=_E2M1_MAG_P).astype(np.uint8)
    sign = (g.random(size=(n, k)) < 0.5).astype(np.uint8) << 3
    c = mag | sign
    packed = (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    sc = g.integers(0x04, 0x10, size=(n, k // 16)).astype(np.uint8)
    return torch.from_numpy(packed), torch.from_numpy(sc)


def hybrid_weights(cfg: HybridConfig, seed: int = 0, random_gains: bool = False,
                   lm_scale: float = 1.0) -> Dict[str, object]:
    """Random-init weights of the hybrid stack.  Linear layers are NVFP4
    (a (codes, scale codes) pair per matrix, [N, K] K-major); the embedding
    is bf16 N(0, 0.02); norm gains 1.0 (or 1 + N(0, 0.1)); conv weights bf16
    N(0, 0.3) [channels, 4] and bias N(0, 0.1); dt_bias U[-6, -2.5], A =
    -U[1, 16], D = N(1, 0.1) in fp32.  ``lm_scale`` multiplies the LM head's
    scales by a power of two (exact) for a peaked variant."""
    g = rng(seed)
    d, I = cfg.d_model, cfg.intermediate
    W: Dict[str, object] = {}
    W["embed"] = normal_bf16(g, (cfg.vocab, d), 0.02)

    def gain(n):
        if random_gains:
            return to_bf16(1.0 + normal_f32(g, (n,), 0.1))
        return to_bf16(np.ones(n, np.float32))

    for l, kind in enumerate(cfg.pattern):
        p = f"l{l}."
        W[p + "norm"] = gain(d)
        if kind == "M":
            W[p + "in_proj"] = nvfp4_weights(g, cfg.in_proj_width, d)
            W[p + "conv_w"] = normal_bf16(g, (cfg.conv_channels, cfg.conv_width), 0.3)
            W[p + "conv_b"] = normal_bf16(g, (cfg.conv_channels,), 0.1)
            W[p + "dt_bias"] = torch.from_numpy(g.uniform(-6.0, -2.5, size=cfg.ssd_heads).astype(np.float32))
            W[p + "A"] = torch.from_numpy((-g.uniform(1.0, 16.0, size=cfg.ssd_heads)).astype(np.float32))
            W[p + "D"] = torch.from_numpy(normal_f32(g, (cfg.ssd_heads,), 0.1, 1.0))
            W[p + "norm_w"] = gain(cfg.d_inner)
            W[p + "out_proj"] = nvfp4_weights(g, d, cfg.d_inner)
        else:
            W[p + "wqkv"] = nvfp4_weights(g, cfg.qkv_width, d)
            W[p + "wo"] = nvfp4_weights(g, d, cfg.q_heads * cfg.head_dim)
        W[p + "mlp_norm"] = gain(d)
        W[p + "wgu"] = nvfp4_weights(g, 2 * I, d)
        W[p + "wd"] = nvfp4_weights(g, d, I)
    W["final_norm"] = gain(d)
    codes, sc = nvfp4_weights(g, cfg.vocab, d)
    if lm_scale != 1.0:
        e = int(round(np.log2(lm_scale)))
        assert 2.0 ** e == lm_scale and 0 <= e <= 4, "lm_scale: a power of two up to 16"
        sc = sc + np.uint8(8 * e)                  # e4m3: +1 in the exponent field doubles
    W["lm_head"] = (codes, sc)
    return W


def hybrid_sequences(cfg: HybridConfig, n: int, lo: int, hi: int, seed: int = 1,
                     prompt_frac: float = 0.75) -> List[Sequence]:
    """n sequences, lengths uniform in [lo, hi], ids uniform; the prompt is
    the first ``prompt_frac`` of each."""
    g = rng(seed)
    out = []
    for _ in range(n):
        L = int(g.integers(lo, hi + 1))
        toks = g.integers(0, cfg.vocab, size=L, dtype=np.int64).astype(np.int32)
        out.append(Sequence(toks, max(1, int(L * prompt_frac))))
    return out


def host_payload(W: Dict[str, object]) -> Dict[str, object]:
    """Raw payloads for the oracle's own decoders: bf16 tensors as uint16
    bits, fp32 as float32 arrays, NVFP4 pairs as (codes, scale codes) uint8."""
    out = {}
    for k, v in W.items():
        if isinstance(v, tuple):
            out[k] = (v[0].numpy().copy(), v[1].numpy().copy())
        elif v.dtype == torch.bfloat16:
            out[k] = bf16_bits(v)
        else:
            out[k] = v.numpy().astype(np.float32).copy()
    return out


def device_nvfp4_weights(gen: torch.Generator, n: int, k: int):
    """The recipe of ``nvfp4_weights`` drawn on the device (packed the same
    way): e2m1 magnitudes from the same categorical distribution (a uniform
    draw located in its cumulative probabilities), a fair sign bit, e4m3 scale
    codes uniform over 0x04..0x0F."""
    dev = gen.device
    cdf = torch.tensor(np.cumsum(_E2M1_MAG_P)[:-1], dtype=torch.float32, device=dev)
    mag = torch.searchsorted(cdf, torch.rand(n, k, generator=gen, device=dev), right=True)
    sign = (torch.rand(n, k, generator=gen, device=dev) < 0.5).to(torch.uint8) << 3
    c = mag.to(torch.uint8) | sign
    packed = c[:, 0::2] | (c[:, 1::2] << 4)
    sc = torch.randint(0x04, 0x10, (n, k // 16), generator=gen, device=dev, dtype=torch.uint8)
    return packed.contiguous(), sc


def device_hybrid_weights(cfg: HybridConfig, seed: int = 0) -> Dict[str, object]:
    """``hybrid_weights``' recipe (unit gains) drawn on the device, for
    throughput runs at full width."""
    gen = device_generator(seed)
    dev = gen.device
    d, I = cfg.d_model, cfg.intermediate
    W: Dict[str, object] = {"embed": device_normal(gen, (cfg.vocab, d), 0.02)}
    ones = lambda n: torch.ones(n, dtype=torch.bfloat16, device=dev)
    for l, kind in enumerate(cfg.pattern):
        p = f"l{l}."
        W[p + "norm"] = ones(d)
        if kind == "M":
            W[p + "in_proj"] = device_nvfp4_weights(gen, cfg.in_proj_width, d)
            W[p + "conv_w"] = device_normal(gen, (cfg.conv_channels, cfg.conv_width), 0.3)
            W[p + "conv_b"] = device_normal(gen, (cfg.conv_channels,), 0.1)
            W[p + "dt_bias"] = torch.rand(cfg.ssd_heads, generator=gen, device=dev) * 3.5 - 6.0
            W[p + "A"] = -(torch.rand(cfg.ssd_heads, generator=gen, device=dev) * 15.0 + 1.0)
            W[p + "D"] = 1.0 + 0.1 * torch.randn(cfg.ssd_heads, generator=gen, device=dev)
            W[p + "norm_w"] = ones(cfg.d_inner)
            W[p + "out_proj"] = device_nvfp4_weights(gen, d, cfg.d_inner)
        else:
            W[p + "wqkv"] = device_nvfp4_weights(gen, cfg.qkv_width, d)
            W[p + "wo"] = device_nvfp4_weights(gen, d, cfg.q_heads * cfg.head_dim)
        W[p + "mlp_norm"] = ones(d)
        W[p + "wgu"] = device_nvfp4_weights(gen, 2 * I, d)
        W[p + "wd"] = device_nvfp4_weights(gen, d, I)
    W["final_norm"] = ones(d)
    W["lm_head"] = device_nvfp4_weights(gen, cfg.vocab, d)
    return W
