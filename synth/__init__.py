"""Seeded synthetic KV-cache workloads (inputs only).

This module produces the inputs that both the CUDA path and the CPU oracle
consume: per-stream generator parameters, calibration tokens, evaluation
tokens and paged block tables.  It holds none of the codec's arithmetic (no
projection, quantisation, packing or bit allocation): it only draws numbers.

Model shapes follow the KV-cache sizes of the models evaluated on the kvtc page
("KV Cache Transform Coding for Compact Storage in LLM Inference", section 1
Problem and section 4 Results: Llama 3.1 8B needs 128 MiB per 1K tokens, i.e.
32 layers x {K,V} x 8 heads x 128 x 2 bytes per token).  No model weights or
datasets are used: each (layer, K|V) stream is low-rank plus noise,

    x_t = mu + A z_t + 0.01 eps_t,   A = Q_D[:, :r] diag(sigma) Q_r^T,
    sigma_i = i^(-p),  z ~ N(0, I_r),  eps ~ N(0, I_D),

with four seeded "outlier" channels multiplied by 10 on K streams where the
workload asks for them, and every value stored as bf16 (round to nearest
even from fp32).

Seeds (numpy PCG64 via ``default_rng``):
  generator parameters  3000 + 2*layer + kv
  calibration tokens    1000 + 2*layer + kv
  evaluation tokens     2000 + 2*layer + kv + 100000*request
  paged block table     4242
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Tuple

import numpy as np

K_STREAM = 0
V_STREAM = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    kv: Tuple[int, ...]          # which of K (0) / V (1) are present
    heads: int
    head_dim: int
    tokens: int                  # tokens per request
    requests: int
    rank: int
    spectrum_p: float
    outliers: bool               # 4 K channels x10
    sink: int
    window: int
    avg_bits: float              # bit budget per coefficient
    group: int = 16
    bmax: int = 8
    n_calib: int = 4096
    block_size: int = 0          # >0: paged restore into blocks of this many tokens
    streamed: bool = False       # layer-by-layer restore on one stream

    @property
    def D(self) -> int:
        return self.heads * self.head_dim

    @property
    def budget_bits(self) -> int:
        return int(round(self.avg_bits * self.D))

    def streams(self) -> List[Tuple[int, int]]:
        """(layer, kv) pairs in storage order: layer-major, K before V."""
        return [(l, kv) for l in range(self.layers) for kv in self.kv]

    def raw_bytes(self) -> int:
        return len(self.streams()) * self.requests * self.tokens * self.D * 2


WORKLOADS = {
    "tiny": Workload("tiny", layers=1, kv=(K_STREAM,), heads=2, head_dim=64,
                     tokens=256, requests=1, rank=32, spectrum_p=1.0,
                     outliers=False, sink=4, window=16, avg_bits=2.0),
    # edge shapes for the kernels' chunking: D an odd multiple of 64 (64-
    # column output chunks, an odd number of 64-wide K blocks) and an odd
    # multiple of 128 (128-column chunks)
    "edge_d192": Workload("edge_d192", layers=1, kv=(0, 1), heads=3,
                          head_dim=64, tokens=700, requests=1, rank=32,
                          spectrum_p=1.0, outliers=True, sink=4, window=16,
                          avg_bits=2.0),
    # 10.42 bits per coefficient: every group at width 8, 256-byte records
    # (the longest the format has)
    "edge_d192_r256": Workload("edge_d192_r256", layers=1, kv=(0, 1),
                               heads=3, head_dim=64, tokens=600, requests=1,
                               rank=32, spectrum_p=1.0, outliers=True, sink=4,
                               window=16, avg_bits=10.42),
    # flat spectrum and 2.5 bits: the DP keeps 15 groups (k = 240, the
    # widest the kernels take)
    "edge_d384": Workload("edge_d384", layers=2, kv=(0, 1), heads=3,
                          head_dim=128, tokens=900, requests=1, rank=384,
                          spectrum_p=0.0, outliers=False, sink=4, window=128,
                          avg_bits=2.5),
    # the widest row the kernels take (D = 8192); 1024-bit budget, 128-byte
    # records; signal rank 224
    "edge_d8192": Workload("edge_d8192", layers=1, kv=(0, 1), heads=64,
                           head_dim=128, tokens=600, requests=1, rank=224,
                           spectrum_p=1.0, outliers=True, sink=4, window=16,
                           avg_bits=0.125),
    "llama31_8b_8k": Workload("llama31_8b_8k", layers=32, kv=(0, 1), heads=8,
                              head_dim=128, tokens=8192, requests=1, rank=128,
                              spectrum_p=1.0, outliers=True, sink=4,
                              window=128, avg_bits=1.0),
    # config-2 shape with a flat spectrum (isotropic latent factors, no
    # outlier channels): the DP keeps 16 two-bit groups, k = 256, the widest
    # the 1-bit/coef budget reaches with this quantiser
    "llama31_8b_8k_flat": Workload("llama31_8b_8k_flat", layers=32,
                                   kv=(0, 1), heads=8, head_dim=128,
                                   tokens=8192, requests=1, rank=1024,
                                   spectrum_p=0.0, outliers=False, sink=4,
                                   window=128, avg_bits=1.0),
    # cross-layer basis: each stream is two consecutive layers of the
    # config-2 shape, a token's rows of layers 2l and 2l + 1 side by side
    # (D = 2 x 8 x 128 = 2048, "layer" l of this workload = that pair), one
    # basis over the pair.  The two layers share their latent factors (rank
    # 128 over the 2048-wide row), the similarity across layers a shared
    # basis relies on; 1 bit per coefficient, as the per-layer workload
    # (256-byte records)
    "llama31_8b_8k_xlayer2": Workload("llama31_8b_8k_xlayer2", layers=16,
                                      kv=(0, 1), heads=16, head_dim=128,
                                      tokens=8192, requests=1, rank=128,
                                      spectrum_p=1.0, outliers=True, sink=4,
                                      window=128, avg_bits=1.0),
    "mistral_nemo_12b_32k": Workload("mistral_nemo_12b_32k", layers=40,
                                     kv=(0, 1), heads=8, head_dim=128,
                                     tokens=32768, requests=1, rank=128,
                                     spectrum_p=1.5, outliers=True, sink=4,
                                     window=128, avg_bits=0.5),
    "llama33_70b_16k": Workload("llama33_70b_16k", layers=80, kv=(0, 1),
                                heads=8, head_dim=128, tokens=16384,
                                requests=1, rank=192, spectrum_p=1.0,
                                outliers=True, sink=4, window=128,
                                avg_bits=1.0, streamed=True),
    "qwen25_7b_paged": Workload("qwen25_7b_paged", layers=28, kv=(0, 1),
                                heads=4, head_dim=128, tokens=4096,
                                requests=64, rank=128, spectrum_p=1.0,
                                outliers=False, sink=4, window=128,
                                avg_bits=2.0, block_size=16),
}


def params_seed(layer: int, kv: int) -> int:
    return 3000 + 2 * layer + kv


def calib_seed(layer: int, kv: int) -> int:
    return 1000 + 2 * layer + kv


def eval_seed(layer: int, kv: int, request: int = 0) -> int:
    return 2000 + 2 * layer + kv + 100000 * request


BLOCK_TABLE_SEED = 4242


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Store generated values as bf16: fp32, then round to nearest even on
    the top 16 bits.  Generated values are finite, so no NaN handling."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


@dataclasses.dataclass
class StreamParams:
    mu: np.ndarray               # [D] fp64
    A: np.ndarray                # [D][r] fp64
    outlier_channels: np.ndarray  # int64 channel ids (empty if none)


def stream_params(w: Workload, layer: int, kv: int) -> StreamParams:
    rng = np.random.default_rng(params_seed(layer, kv))
    D, r = w.D, w.rank
    mu = rng.standard_normal(D)
    qd, _ = np.linalg.qr(rng.standard_normal((D, r)))
    qr_, _ = np.linalg.qr(rng.standard_normal((r, r)))
    sigma = np.arange(1, r + 1, dtype=np.float64) ** (-w.spectrum_p)
    A = (qd * sigma) @ qr_.T
    if w.outliers and kv == K_STREAM:
        ch = np.sort(rng.choice(D, size=4, replace=False)).astype(np.int64)
    else:
        ch = np.zeros(0, dtype=np.int64)
    return StreamParams(mu, A, ch)


def _draw(p: StreamParams, rng: np.random.Generator, n: int) -> np.ndarray:
    D, r = p.A.shape
    z = rng.standard_normal((n, r))
    eps = rng.standard_normal((n, D))
    x = p.mu[None, :] + z @ p.A.T + 0.01 * eps
    if p.outlier_channels.size:
        x[:, p.outlier_channels] *= 10.0
    return f32_to_bf16_bits(x)


def calib_tokens(w: Workload, layer: int, kv: int,
                 params: Optional[StreamParams] = None) -> np.ndarray:
    """Calibration tokens, bf16 bits [n_calib][D]."""
    p = params if params is not None else stream_params(w, layer, kv)
    return _draw(p, np.random.default_rng(calib_seed(layer, kv)), w.n_calib)


def eval_tokens(w: Workload, layer: int, kv: int, request: int = 0,
                T: Optional[int] = None,
                params: Optional[StreamParams] = None) -> np.ndarray:
    """Evaluation tokens of one request, bf16 bits [T][D] (numpy)."""
    p = params if params is not None else stream_params(w, layer, kv)
    n = w.tokens if T is None else T
    return _draw(p, np.random.default_rng(eval_seed(layer, kv, request)), n)


def eval_tokens_torch(w: Workload, layer: int, kv: int, request: int = 0,
                      T: Optional[int] = None, device="cuda",
                      params: Optional[StreamParams] = None):
    """Same recipe drawn with torch's generator on ``device`` (fast for the
    multi-GB workloads).  The numbers differ from :func:`eval_tokens` (another
    generator) but the distribution and seed are the same.  Returns a bf16
    tensor [T][D]."""
    p = params if params is not None else stream_params(w, layer, kv)
    n = w.tokens if T is None else T
    return _draw_torch(p, eval_seed(layer, kv, request), n, device)


def calib_tokens_torch(w: Workload, layer: int, kv: int, device="cuda",
                       params: Optional[StreamParams] = None):
    """Calibration tokens drawn with torch's generator on ``device`` (same
    recipe and seed as :func:`calib_tokens`, other generator); bf16
    [n_calib][D]."""
    return _draw_torch(stream_params(w, layer, kv) if params is None
                       else params, calib_seed(layer, kv), w.n_calib, device)


def _draw_torch(p: StreamParams, seed: int, n: int, device):
    import torch
    D, r = p.A.shape
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    z = torch.randn((n, r), generator=g, device=device, dtype=torch.float32)
    eps = torch.randn((n, D), generator=g, device=device, dtype=torch.float32)
    A = torch.from_numpy(p.A.astype(np.float32)).to(device)
    mu = torch.from_numpy(p.mu.astype(np.float32)).to(device)
    x = torch.addmm(mu[None, :], z, A.T)
    x.add_(eps, alpha=0.01)
    if p.outlier_channels.size:
        ch = torch.from_numpy(p.outlier_channels).to(device)
        x[:, ch] *= 10.0
    return x.to(torch.bfloat16)


def block_table(w: Workload) -> np.ndarray:
    """Paged layout: a seeded random permutation of all physical blocks,
    int32 [requests][blocks_per_request]."""
    assert w.block_size > 0
    per_req = -(-w.tokens // w.block_size)
    rng = np.random.default_rng(BLOCK_TABLE_SEED)
    perm = rng.permutation(w.requests * per_req).astype(np.int32)
    return perm.reshape(w.requests, per_req)
