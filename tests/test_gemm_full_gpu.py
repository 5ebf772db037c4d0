"""The verify / prefill GEMM (self-speculative verify: "ntransformer - moteur
d'inférence NVMe-to-GPU…", "Fonctionnalités principales"; prompt chunks: KV
cache) at full size, in the launch configuration the benchmark times
(nt_gemm_q on a plain x, the GEMM workloads' seeds): the two timed GEMM
workloads and the 8B prompt-chunk shapes with 16 vectors.  Sampled rows —
random ones plus the edges of the first and last 16-row tiles — against the
fp64 oracle one by one, and every row against the decode GEMV of the same
vector (itself pinned to the oracle at full size), each within the GEMV
bound (relative L2 1e-3)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import dev, host, need_gpu, rel_l2, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    from block_quantized_gemv_nt_gb300 import nt
    c = nt.Context(0)
    yield c
    c.sync()
    c.close()


@pytest.mark.parametrize("fmt,rows,cols,M", [
    (synth.Q8_0, 14336, 4096, 8),    # gemm_q8_0_14336x4096_m8
    (synth.Q6_K, 8192, 28672, 5),    # gemm_q6_k_8192x28672_m5
    (synth.Q8_0, 6144, 4096, 16),    # 8B Q/K/V over a 16-token prompt chunk
    (synth.Q8_0, 4096, 14336, 16),   # 8B down projection, 16 tokens
    (synth.Q4_K, 28672, 8192, 16),   # 70B Q4_K_M gate / up, 16 tokens
])
def test_gemm_full_size(ctx, fmt, rows, cols, M):
    from block_quantized_gemv_nt_gb300 import nt
    seed = 100 + fmt
    W = synth.quant_matrix(fmt, rows, cols, seed=seed, stream=0)
    X = synth.normal_f32(M * cols, seed=seed, stream=1).reshape(M, cols)
    Wd, Xd = dev(W), dev(X)
    Y = torch.empty(M, rows, dtype=torch.float32, device="cuda")
    nt.nt_gemm_q(ctx, fmt, Wd, Xd, Y, rows, cols, M)
    torch.cuda.synchronize()
    Yh = host(Y)
    rng = np.random.default_rng(seed)
    idx = np.unique(np.concatenate([rng.choice(rows, 240, replace=False),
                                    [0, 15, 16, rows - 17, rows - 16, rows - 1]]))
    Ws = np.ascontiguousarray(W[idx])
    y1 = torch.empty(rows, dtype=torch.float32, device="cuda")
    for m in range(M):
        ref = oracle.gemv(fmt, Ws, X[m].astype(np.float64), len(idx), cols)
        assert rel_l2(Yh[m, idx], ref) <= 1e-3, m
        nt.nt_gemv_q(ctx, fmt, Wd, Xd[m], y1, rows, cols)
        torch.cuda.synchronize()
        assert rel_l2(Yh[m], host(y1).astype(np.float64)) <= 1e-3, m
