"""Workload shapes and seeded input tensors for CSA / HCA layers.

The five workloads below are the synthetic configurations the method is measured on: a tiny
CSA+HCA prefill pair, CSA decode at 128K context, HCA decode at 1M context, a CSA prefill chunk of
8192 queries against 128K context, and a CSA/HCA decode pair at 1M context.

Distributions (every tensor has its own generator stream, keyed by seed, layer and tensor id):
  * Q            ~ N(0,1) * q_scale, rounded to bf16 (q_scale = 1/sqrt(d) folds the softmax scale)
  * raw K, raw V ~ N(0,1), rounded to bf16
  * pooling logits w ~ N(0,1), fp32, one per token
  * indexer codes: bytes uniform on [0,255] (two e2m1 codes per byte, each uniform on 16 codes)
  * indexer scales: UE8M0 bytes uniform on {123..127} (2^-4 .. 2^0)
Nothing here computes any part of the method.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class LayerShape:
    kind: str            # "csa" or "hca"
    B: int               # sequences
    N: int               # context tokens, including the queries' own tokens
    Nq: int              # query tokens per sequence (positions q_pos0 .. q_pos0+Nq-1)
    q_pos0: int
    H: int               # query heads (one shared KV head)
    d: int               # head dim
    m: int               # tokens per compressed entry (4 for CSA, 128 for HCA)
    W: int               # sliding-window length in raw tokens
    k: int = 0           # CSA top-k (0 for HCA)
    H_I: int = 0         # indexer heads (CSA)
    d_I: int = 0         # indexer dim (CSA)
    q_scale: float = 0.0 # multiplier on N(0,1) queries
    compress_begin: int = 0  # first token whose block is compressed inside the step

    @property
    def E(self) -> int:
        return self.N // self.m

    def scaled(self, **kw) -> "LayerShape":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    description: str
    seed: int
    layers: Tuple[LayerShape, ...]
    mode: str            # "decode" or "prefill"

    def layer(self, kind: str) -> LayerShape:
        for l in self.layers:
            if l.kind == kind:
                return l
        raise KeyError(kind)


def _decode_layer(kind, B, N, H, d, m, W, k=0, H_I=0, d_I=0) -> LayerShape:
    return LayerShape(kind=kind, B=B, N=N, Nq=1, q_pos0=N - 1, H=H, d=d, m=m, W=W, k=k,
                      H_I=H_I, d_I=d_I, q_scale=1.0 / math.sqrt(d), compress_begin=N - m)


CONFIGS: Dict[str, Workload] = {}


def _add(w: Workload) -> None:
    CONFIGS[w.name] = w


_add(Workload(
    name="tiny_pair_prefill_2k",
    description="CSA+HCA layer pair, prefill, batch 1, seq 2048, 8 heads x 64, "
                "CSA block 4 top-k 64 window 64 (indexer 2 heads x 32), HCA block 128 window 64",
    seed=0, mode="prefill",
    layers=(
        LayerShape("csa", B=1, N=2048, Nq=2048, q_pos0=0, H=8, d=64, m=4, W=64, k=64,
                   H_I=2, d_I=32, q_scale=1.0 / 8.0, compress_begin=0),
        LayerShape("hca", B=1, N=2048, Nq=2048, q_pos0=0, H=8, d=64, m=128, W=64,
                   q_scale=1.0 / 8.0, compress_begin=0),
    )))

_add(Workload(
    name="csa_decode_128k",
    description="CSA decode step, batch 16, context 131072 (32768 entries), 64 heads x 128, "
                "indexer 4 heads x 64 FP4, top-k 512, window 128",
    seed=1, mode="decode",
    layers=(_decode_layer("csa", B=16, N=131072, H=64, d=128, m=4, W=128, k=512, H_I=4, d_I=64),)))

_add(Workload(
    name="hca_decode_1m",
    description="HCA decode step, batch 32, context 1048576 (8192 entries), 64 heads x 128, "
                "window 128",
    seed=2, mode="decode",
    layers=(_decode_layer("hca", B=32, N=1048576, H=64, d=128, m=128, W=128),)))

_add(Workload(
    name="csa_prefill_8k_of_128k",
    description="CSA prefill chunk of 8192 queries against a 131072-token causal context, "
                "block-4 compression of the chunk's tokens, 64 heads x 128, indexer 4 x 64 FP4, "
                "top-k 2048, window 128",
    seed=3, mode="prefill",
    layers=(LayerShape("csa", B=1, N=131072, Nq=8192, q_pos0=131072 - 8192, H=64, d=128, m=4,
                       W=128, k=2048, H_I=4, d_I=64, q_scale=1.0 / math.sqrt(128),
                       compress_begin=131072 - 8192),)))

_add(Workload(
    name="pair_decode_1m",
    description="CSA/HCA layer pair decode, batch 4, context 1048576: CSA 262144 entries "
                "(indexer 4 x 64 FP4, top-k 2048), HCA 8192 entries, 64 heads x 128, window 128",
    seed=4, mode="decode",
    layers=(
        _decode_layer("csa", B=4, N=1048576, H=64, d=128, m=4, W=128, k=2048, H_I=4, d_I=64),
        _decode_layer("hca", B=4, N=1048576, H=64, d=128, m=128, W=128),
    )))

# Short aliases by position in the table above (1-based).
_ORDER = list(CONFIGS)


def get_config(name_or_index) -> Workload:
    if isinstance(name_or_index, int) or str(name_or_index).isdigit():
        return CONFIGS[_ORDER[int(name_or_index) - 1]]
    return CONFIGS[name_or_index]


_TENSOR_IDS = {"q": 1, "k_raw": 2, "v_raw": 3, "logits": 4,
               "qi_codes": 5, "qi_scales": 6, "ki_codes": 7, "ki_scales": 8, "xi_raw": 9}


def _gen(seed: int, layer_id: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) << 20) ^ (int(layer_id) << 8) ^ _TENSOR_IDS[name])
    return g


def _normal_bf16(shape, scale, g, device, rows_per_chunk=1 << 20) -> torch.Tensor:
    """N(0,1)*scale rounded to bf16, drawn in row chunks so a 1M-token cache needs no
    full-size fp32 temporary."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1, shape[-1])
    for r0 in range(0, flat.shape[0], rows_per_chunk):
        r1 = min(flat.shape[0], r0 + rows_per_chunk)
        t = torch.randn((r1 - r0, shape[-1]), generator=g, device=device, dtype=torch.float32)
        if scale != 1.0:
            t.mul_(scale)
        flat[r0:r1].copy_(t)
    return out


def generate_layer(shape: LayerShape, seed: int, layer_id: int = 0,
                   device: Optional[torch.device] = None,
                   skip: Tuple[str, ...] = ()) -> Dict[str, torch.Tensor]:
    """Draw every input tensor of one layer on `device` (bf16 as torch.bfloat16, codes and
    scales as uint8, logits as float32). Layouts are row-major:
      q [B,Nq,H,d]; k_raw,v_raw [B,N,d]; logits [B,N];
      qi_codes [B,Nq,H_I,d_I/2]; qi_scales [B,Nq,H_I,d_I/32];
      ki_codes [B,E,d_I/2]; ki_scales [B,E,d_I/32]  (CSA only)."""
    device = torch.device(device) if device is not None else torch.device("cpu")
    s = shape
    out: Dict[str, torch.Tensor] = {}
    if "q" not in skip:
        out["q"] = _normal_bf16((s.B, s.Nq, s.H, s.d), s.q_scale, _gen(seed, layer_id, "q", device), device)
    if "k_raw" not in skip:
        out["k_raw"] = _normal_bf16((s.B, s.N, s.d), 1.0, _gen(seed, layer_id, "k_raw", device), device)
    if "v_raw" not in skip:
        out["v_raw"] = _normal_bf16((s.B, s.N, s.d), 1.0, _gen(seed, layer_id, "v_raw", device), device)
    if "logits" not in skip:
        out["logits"] = torch.randn((s.B, s.N), generator=_gen(seed, layer_id, "logits", device),
                                    device=device, dtype=torch.float32)
    if s.kind == "csa":
        assert s.d_I % 32 == 0 and s.H_I > 0
        E = s.E
        out["qi_codes"] = torch.randint(0, 256, (s.B, s.Nq, s.H_I, s.d_I // 2),
                                        generator=_gen(seed, layer_id, "qi_codes", device),
                                        device=device, dtype=torch.uint8)
        out["qi_scales"] = torch.randint(123, 128, (s.B, s.Nq, s.H_I, s.d_I // 32),
                                         generator=_gen(seed, layer_id, "qi_scales", device),
                                         device=device, dtype=torch.uint8)
        out["ki_codes"] = torch.randint(0, 256, (s.B, E, s.d_I // 2),
                                        generator=_gen(seed, layer_id, "ki_codes", device),
                                        device=device, dtype=torch.uint8)
        out["ki_scales"] = torch.randint(123, 128, (s.B, E, s.d_I // 32),
                                         generator=_gen(seed, layer_id, "ki_scales", device),
                                         device=device, dtype=torch.uint8)
    return out


def index_key_rows(shape: LayerShape, seed: int, layer_id: int = 0,
                   device: Optional[torch.device] = None) -> torch.Tensor:
    """Per-token index-key rows xi_raw [B, N, d_I], N(0,1) rounded to bf16 (the input the
    indexer's own compressed keys are pooled from)."""
    device = torch.device(device) if device is not None else torch.device("cpu")
    s = shape
    return _normal_bf16((s.B, s.N, s.d_I), 1.0, _gen(seed, layer_id, "xi_raw", device), device)


def bf16_bits(t: torch.Tensor):
    """Host numpy uint16 view of a bf16 tensor's bits (for the oracle)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")
