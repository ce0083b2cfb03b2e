"""Full-size workloads on the GPU, checked against the oracle.

At these sizes the oracle computes every INT8 code and scale in full (bit
exact) and the contraction plus dequant at sampled output positions (the
four corners of every problem, the last row and column, and random
positions), which it evaluates one by one.  The GPU runs each workload the
way the benchmark does: weights quantized on the GPU, then the whole layer
through ``linear`` (per-token quantization into the workspace, then GEMM for
M > 1 or the matrix-vector kernel for M == 1).

Workloads (seed 0; recipes in w4a8_int8_quantized_gb300.synth):
  * per-channel sweep, N=10240, K=2560, M in {1, 128, 1024, 4096, 8192},
    x ~ N(0,1) with 26 of 2560 K-channels x30;
  * per-group gs=128 and gs=64, N=10240, K=2560, M=4096, heavy-tailed rows;
  * W4A8, N=14336, K=4096, M in {1, 2048};
  * the four linear layers of an 8B-class decoder block at M=4516 and M=1,
    inputs with 6 outlier channels x50.
"""
import numpy as np
import pytest

import oracle
from w4a8_int8_quantized_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import w4a8_int8_quantized_gb300 as w8

from test_gpu_parity import assert_bits, assert_fp16_close, dev, host  # noqa: E402


def sample_positions(M, N, count=3000, seed=0):
    rng = np.random.default_rng(seed)
    rows = list(rng.integers(0, M, count)) + [0, 0, M - 1, M - 1] + [M - 1] * 8 + list(range(min(M, 8)))
    cols = list(rng.integers(0, N, count)) + [0, N - 1, 0, N - 1] + list(range(N - 8, N)) + [N - 1] * min(M, 8)
    return np.array(rows, np.int64), np.array(cols, np.int64)


def run_layer(x, W, gs=0, wbits=8, check_i32=True, exact=True):
    M, K = x.shape
    N = W.shape[0]
    xd, Wd = dev(x), dev(W)
    if wbits == 8:
        wq, sw = w8.quantize_weight_int8(Wd, gs)
        rq, rs = oracle.quantize_weight_int8(W, gs)
        rw = rq
    else:
        wq, sw = w8.pack_weight_int4(Wd)
        rq, rs = oracle.pack_weight_int4(W)
        rw = oracle.unpack_int4(rq, K)
    np.testing.assert_array_equal(host(wq), rq)
    np.testing.assert_array_equal(host(sw), rs)
    del Wd
    y = w8.linear(xd, wq, sw, gs, wbits)
    xq, sa = w8.quantize_act_per_token(xd, gs)
    rxq, rsa = oracle.quantize_act_per_token(x, gs)
    np.testing.assert_array_equal(host(xq), rxq)
    np.testing.assert_array_equal(host(sa), rsa)
    rows, cols = sample_positions(M, N)
    racc, ry = oracle.sampled_outputs(rxq, rsa, rw, rs, rows, cols, gs)
    rt, ct = torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()
    ys = host(y[rt, ct])
    # tolerance scale from the sampled reference (max|y| over the samples)
    assert_fp16_close(ys, ry)
    if exact:
        assert_bits(ys, ry)
    if check_i32 and M > 1:
        acc = w8.w8a8_gemm_i32(xq, wq, gs, wbits)
        np.testing.assert_array_equal(host(acc[rt, ct]), racc)
        del acc
    del y, xq, sa, wq, sw, xd
    torch.cuda.empty_cache()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    w8.load()


@pytest.mark.parametrize("M", synth.WORKLOADS["pc_sweep"]["Ms"])
def test_per_channel_sweep(M):
    cfg = synth.WORKLOADS["pc_sweep"]
    x = synth.activations(M, cfg["K"], seed=0, **cfg["act"])
    W = synth.weights(cfg["N"], cfg["K"], seed=0)
    run_layer(x, W)


@pytest.mark.parametrize("gs", synth.WORKLOADS["pg"]["gs"])
def test_per_group(gs):
    cfg = synth.WORKLOADS["pg"]
    M = cfg["Ms"][0]
    x = synth.activations(M, cfg["K"], seed=0, **cfg["act"])
    W = synth.weights(cfg["N"], cfg["K"], seed=0)
    run_layer(x, W, gs=gs, exact=False)


@pytest.mark.parametrize("M", synth.WORKLOADS["w4a8"]["Ms"])
def test_w4a8(M):
    cfg = synth.WORKLOADS["w4a8"]
    x = synth.activations(M, cfg["K"], seed=0, **cfg["act"])
    W = synth.weights(cfg["N"], cfg["K"], seed=0)
    run_layer(x, W, wbits=4)


@pytest.mark.parametrize("layer", [l[0] for l in synth.BLOCK_LAYERS])
@pytest.mark.parametrize("M", synth.BLOCK_MS)
def test_decoder_block_layers(layer, M):
    name, N, K = next(l for l in synth.BLOCK_LAYERS if l[0] == layer)
    x = synth.activations(M, K, seed=0, salt=K, **synth.BLOCK_ACT)
    W = synth.weights(N, K, seed=0, salt=N)
    run_layer(x, W)
