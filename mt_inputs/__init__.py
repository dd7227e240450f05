"""Seeded synthetic inputs for the layer-streamed decoder training step.

This module is shared by the test harness, the oracle side and the product
side, so it holds none of the method's arithmetic: it only names the workload
shapes and draws the random weights and tokens that both sides then consume.

Recipe (the MegaTrain pages fine-tune Qwen2.5-7B/14B-shaped decoders on
MetaMathQA; neither the dataset nor trained weights exist here, so uniform
random tokens and N(0, 0.02) weights stand in for them):

* weights of tile k (0 = embedding, 1..L = decoder layers, L+1 = head) come
  from ``torch.Generator().manual_seed(1000 + k)``: each matrix is
  ``randn(fp32) * 0.02`` rounded to BF16 (round-to-nearest-even, torch's cast);
  RMSNorm gains are ones (or ``1 + jitter * randn`` when a test asks for
  jitter, to make a dropped gain visible);
* tokens of step n come from ``manual_seed(2000 + n)``: ``randint(0, V)``
  int32 of shape [B, S + 1]; row b feeds ``tokens[b, :S]`` and predicts
  ``tokens[b, 1:]``.

Per-tile seeds let any single layer be regenerated without the rest.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace

import torch

__all__ = [
    "ModelShape",
    "PRESETS",
    "layer_tensor_shapes",
    "embed_weights",
    "layer_weights",
    "head_weights",
    "model_weights",
    "step_tokens",
    "normal_bf16",
]


@dataclass(frozen=True)
class ModelShape:
    """Shape and hyper-parameters of one Llama-style decoder workload."""

    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    batch: int
    seq: int
    ckpt_every: int = 1
    rms_eps: float = 1e-5
    rope_theta: float = 1e4
    lr: float = 1e-4
    beta1: float = 0.9
    beta2: float = 0.95
    adam_eps: float = 1e-8
    weight_decay: float = 0.0
    n_experts: int = 0  # > 0: every layer's MLP is a top_k mixture of n_experts SwiGLU experts of width ffn
    top_k: int = 0

    def with_(self, **kw) -> "ModelShape":
        return replace(self, **kw)

    @property
    def tokens_per_step(self) -> int:
        return self.batch * self.seq


# Workloads: the tiny decoder, the ~1.3B decoder, the 14B-shaped GQA decoder,
# the 70B-shaped GQA decoder and the long-context 7B decoder (seq swept).
PRESETS = {
    "tiny": ModelShape("tiny", 2, 256, 4, 4, 64, 688, 1024, 2, 128, ckpt_every=1),
    "1.3b": ModelShape("1.3b", 24, 2048, 16, 16, 128, 5632, 32000, 8, 2048, ckpt_every=2),
    "14b": ModelShape("14b", 48, 5120, 40, 8, 128, 13824, 152064, 8, 4096, ckpt_every=1),
    "70b": ModelShape("70b", 80, 8192, 64, 8, 128, 28672, 128256, 4, 4096, ckpt_every=1),
    "7b-32k": ModelShape("7b-32k", 32, 4096, 32, 32, 128, 11008, 32000, 1, 32768, ckpt_every=1),
    "7b-128k": ModelShape("7b-128k", 32, 4096, 32, 32, 128, 11008, 32000, 1, 131072, ckpt_every=1),
    "7b-512k": ModelShape("7b-512k", 32, 4096, 32, 32, 128, 11008, 32000, 1, 524288, ckpt_every=1),
}

LAYER_TENSORS = ("g1", "wq", "wk", "wv", "wo", "g2", "wg", "wu", "wd")


def layer_tensor_shapes(s: ModelShape) -> dict:
    """Named decoder-layer tensors in nn.Linear [out, in] convention."""
    q = s.n_heads * s.head_dim
    kv = s.n_kv_heads * s.head_dim
    return {
        "g1": (s.d_model,),
        "wq": (q, s.d_model),
        "wk": (kv, s.d_model),
        "wv": (kv, s.d_model),
        "wo": (s.d_model, q),
        "g2": (s.d_model,),
        "wg": (s.ffn, s.d_model),
        "wu": (s.ffn, s.d_model),
        "wd": (s.d_model, s.ffn),
    }


def _matrix(gen: torch.Generator, shape, std: float = 0.02) -> torch.Tensor:
    return (torch.randn(shape, generator=gen, dtype=torch.float32) * std).to(torch.bfloat16)


def _gain(gen: torch.Generator, n: int, jitter: float) -> torch.Tensor:
    if jitter == 0.0:
        return torch.ones(n, dtype=torch.bfloat16)
    return (1.0 + jitter * torch.randn(n, generator=gen, dtype=torch.float32)).to(torch.bfloat16)


def embed_weights(s: ModelShape) -> dict:
    gen = torch.Generator().manual_seed(1000)
    return {"E": _matrix(gen, (s.vocab, s.d_model))}


def layer_weights(s: ModelShape, layer: int, gain_jitter: float = 0.0) -> dict:
    """Weights of decoder layer ``layer`` (0-based; tile index layer + 1)."""
    gen = torch.Generator().manual_seed(1000 + layer + 1)
    out = {}
    for name, shape in layer_tensor_shapes(s).items():
        if name in ("g1", "g2"):
            out[name] = _gain(gen, shape[0], gain_jitter)
        else:
            out[name] = _matrix(gen, shape)
    return out


def moe_layer_weights(s: ModelShape, layer: int, gain_jitter: float = 0.0) -> dict:
    """Weights of MoE decoder layer ``layer``: the attention half as in
    ``layer_weights``, the router ``wr`` [E, d] and ``experts``, a list of
    {'wg', 'wu' [ffn, d], 'wd' [d, ffn]}."""
    gen = torch.Generator().manual_seed(5000 + layer + 1)
    dense = layer_weights(s, layer, gain_jitter)
    out = {k: dense[k] for k in ("g1", "wq", "wk", "wv", "wo", "g2")}
    out["wr"] = _matrix(gen, (s.n_experts, s.d_model), std=0.2)
    out["experts"] = [{"wg": _matrix(gen, (s.ffn, s.d_model)), "wu": _matrix(gen, (s.ffn, s.d_model)),
                       "wd": _matrix(gen, (s.d_model, s.ffn))} for _ in range(s.n_experts)]
    return out


def head_weights(s: ModelShape, gain_jitter: float = 0.0) -> dict:
    gen = torch.Generator().manual_seed(1000 + s.n_layers + 1)
    return {"gf": _gain(gen, s.d_model, gain_jitter), "wh": _matrix(gen, (s.vocab, s.d_model))}


def model_weights(s: ModelShape, gain_jitter: float = 0.0) -> dict:
    """All BF16 weights: {'embed': {...}, 'layers': [{...}, ...], 'head': {...}}."""
    return {
        "embed": embed_weights(s),
        "layers": [(moe_layer_weights if s.n_experts else layer_weights)(s, i, gain_jitter)
                   for i in range(s.n_layers)],
        "head": head_weights(s, gain_jitter),
    }


def tied(params: dict) -> dict:
    """The same weights with the LM head tied to the embedding: ``head`` keeps
    only the final norm gain and the embedding E serves as the head's weight."""
    return {"embed": params["embed"], "layers": params["layers"], "head": {"gf": params["head"]["gf"]}}


def step_tokens(s: ModelShape, step: int) -> torch.Tensor:
    """int32 [B, S+1] uniform token ids for training step ``step`` (1-based)."""
    gen = torch.Generator().manual_seed(2000 + step)
    return torch.randint(0, s.vocab, (s.batch, s.seq + 1), generator=gen, dtype=torch.int64).to(torch.int32)


def normal_bf16(shape, seed: int, std: float = 1.0, chunk: int = 1 << 24) -> torch.Tensor:
    """Large BF16 arrays of N(0, std^2) values (activations, output gradients).

    The flat array is cut into chunks of ``chunk`` elements; chunk c is
    ``randn(fp32, generator seeded with seed * 1_000_003 + c) * std`` rounded
    to BF16, drawn on parallel threads.  The values depend only on (shape,
    seed, std, chunk).
    """
    n = 1
    for x in shape:
        n *= int(x)
    out = torch.empty(n, dtype=torch.bfloat16)

    def fill(c):
        lo = c * chunk
        hi = min(n, lo + chunk)
        g = torch.Generator().manual_seed(seed * 1_000_003 + c)
        out[lo:hi] = (torch.randn(hi - lo, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)

    with ThreadPoolExecutor(max_workers=max(1, min(16, torch.get_num_threads()))) as ex:
        list(ex.map(fill, range((n + chunk - 1) // chunk)))
    return out.reshape(shape)
