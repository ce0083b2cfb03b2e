"""Seeded synthetic inputs for the quantized linear layer.

This module only draws random fp16 tensors with the shapes and value
distributions of the workloads; it holds none of the method's arithmetic
(no quantization, no contraction).  Both the tests (CUDA path and oracle)
and the benchmark take their inputs from here, so the two sides see the same
bytes.

Recipe (numpy PCG64, one independent sub-stream per tensor):

* activations x [M, K] fp16: N(0, 1); optionally ``n_outliers`` K-channels
  (the same channels for every row, drawn without replacement) multiplied by
  ``outlier_scale``; optionally heavy-tailed rows x[m, :] = z[m, :] * |t_3|
  with one Student-t (3 degrees of freedom) draw per row;
* weights W [N, K] fp16: N(0, 0.02^2).
"""
from __future__ import annotations

import numpy as np

_STREAM_X, _STREAM_W, _STREAM_OUTLIER, _STREAM_ROWS = 1, 2, 3, 4


def _rng(seed: int, stream: int, salt: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, salt])))


def activations(M: int, K: int, seed: int = 0, n_outliers: int = 0,
                outlier_scale: float = 1.0, heavy_rows: bool = False,
                salt: int = 0) -> np.ndarray:
    z = _rng(seed, _STREAM_X, salt).standard_normal((M, K), dtype=np.float32)
    if n_outliers:
        ch = _rng(seed, _STREAM_OUTLIER, salt).choice(K, size=n_outliers, replace=False)
        z[:, ch] *= np.float32(outlier_scale)
    if heavy_rows:
        r = np.abs(_rng(seed, _STREAM_ROWS, salt).standard_t(3, size=(M, 1))).astype(np.float32)
        z *= r
    return z.astype(np.float16)


def weights(N: int, K: int, seed: int = 0, std: float = 0.02, salt: int = 0) -> np.ndarray:
    w = _rng(seed, _STREAM_W, salt).standard_normal((N, K), dtype=np.float32)
    w *= np.float32(std)
    return w.astype(np.float16)


# Workload recipes: (name, M list, N, K, group sizes, wbits, activation kwargs).
WORKLOADS = {
    # W8A8 per-channel, small: 4 of 512 K-channels scaled x40.
    "pc_small": dict(Ms=[128], N=512, K=512, gs=[0], wbits=8,
                     act=dict(n_outliers=4, outlier_scale=40.0)),
    # W8A8 per-channel shape sweep, N=10240, K=2560; 1% of K-channels x30.
    "pc_sweep": dict(Ms=[1, 128, 1024, 4096, 8192], N=10240, K=2560, gs=[0], wbits=8,
                     act=dict(n_outliers=26, outlier_scale=30.0)),
    # W8A8 per-group gs=128 and gs=64, heavy-tailed rows.
    "pg": dict(Ms=[4096], N=10240, K=2560, gs=[128, 64], wbits=8,
               act=dict(heavy_rows=True)),
    # W4A8 per-channel, N=14336, K=4096.
    "w4a8": dict(Ms=[1, 2048], N=14336, K=4096, gs=[0], wbits=4, act=dict()),
}

# The linear layers of one 8B-class decoder block (hidden 4096, 32 q / 8 kv
# heads of dim 128, intermediate 14336), as (name, N, K); W8A8 per-channel,
# inputs with 6 outlier channels x50, prefill M=4516 plus decode M=1.
BLOCK_LAYERS = [("qkv", 6144, 4096), ("o_proj", 4096, 4096),
                ("gate_up", 28672, 4096), ("down", 4096, 14336)]
BLOCK_ACT = dict(n_outliers=6, outlier_scale=50.0)
BLOCK_MS = [4516, 1]
