"""GPU parity of the routing kernels (bit-exact against the oracle on the same fp32 logits)
and of the tensor-core GEMM building block (against a float64 matmul)."""
import numpy as np
import pytest
import torch

from latent_compressed_expert_gb300 import lmoe, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from latent_compressed_expert_gb300 import build
    build.build()
    lmoe.load()
    return torch.device("cuda:0")


# ----------------------------------------------------------------------------------------
# tcgen05 GEMM
# ----------------------------------------------------------------------------------------
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 256, 128), (1, 16, 64), (300, 640, 448),
                                   (513, 384, 1024), (64, 896, 3584), (1000, 1280, 512),
                                   (4096, 512, 256),
                                   # tile pairs (two M-tiles per CTA), 256- and 128-wide tiles;
                                   # M ragged, the last pair's second tile wholly past M
                                   (20000, 3584, 2048), (26000, 384, 2048),
                                   # 256 x 256 tiles over SM pairs with N ragged: the last
                                   # tile's 16 valid columns all in rank 0's half of B
                                   (20000, 2832, 2048),
                                   # the same with GEMM 1's reduction length (K = 7168)
                                   (8192, 2560, 7168),
                                   # 224-wide tiles (N = 896 and 672), single and paired;
                                   # over SM pairs at 5000 rows, the last cluster tile's
                                   # second 128 rows holding 8
                                   (8192, 896, 3584), (300, 672, 512), (20000, 896, 2048),
                                   (5000, 896, 3584)])
def test_gemm_matches_float64(dev, M, N, K):
    g = torch.Generator(device=dev).manual_seed(M * 7 + N * 3 + K)
    A = torch.randn(M, K, generator=g, device=dev).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g, device=dev).to(torch.bfloat16)
    C, flag = lmoe.gemm_bf16(A, B)
    torch.cuda.synchronize()
    assert int(flag[0]) == 0
    ref = A.double() @ B.double().T
    bound = K * 2.0 ** -23 * (A.double().abs() @ B.double().abs().T) + 1e-30
    err = (C.double() - ref).abs()
    assert bool((err <= bound).all()), float((err / bound).max())


@pytest.mark.parametrize("M,N,T", [
    # one-SM tiles (grouped-K mode, one group): ragged T, M below one tile, N ragged
    (128, 256, 64), (200, 512, 1000), (1024, 3584, 146),
    # 256 x 256 cluster tiles over SM pairs (at least two per SM pair): T ragged, M and N ragged
    # across the pair, and T = 8192 as in the K3 prefill weight gradients
    (4096, 5120, 1000), (4104, 5136, 777), (7168, 7680, 8192)])
def test_weight_gradient_gemm_matches_float64(dev, M, N, T):
    """C = A^T B over all T rows, the backward's weight-gradient form, against float64."""
    g = torch.Generator(device=dev).manual_seed(M * 5 + N * 3 + T)
    A = torch.randn(T, M, generator=g, device=dev).to(torch.bfloat16)
    B = torch.randn(T, N, generator=g, device=dev).to(torch.bfloat16)
    C, words = lmoe.gemm_wgrad_bf16(A, B)
    torch.cuda.synchronize()
    assert int(words[0]) == 0
    ref = A.double().T @ B.double()
    bound = max(T, 1) * 2.0 ** -23 * (A.double().abs().T @ B.double().abs()) + 1e-30
    err = (C.double() - ref).abs()
    assert bool((err <= bound).all()), float((err / bound).max())



# ----------------------------------------------------------------------------------------
# routing: bit-exact against the oracle on identical fp32 logits
# ----------------------------------------------------------------------------------------
def _logits(T, E, kind, seed):
    if kind == "normal":
        return synth.make_logits(T, E, seed)
    if kind == "ties":
        return synth.make_uniform_logits(T, E, seed, quantum=0.25)
    if kind == "saturated":          # many scores round to exactly 1.0 (and to ~0)
        return synth.make_logits(T, E, seed, scale=30.0)
    if kind == "zipf":
        return synth.make_logits(T, E, seed, zipf_s=1.1)
    raise ValueError(kind)


ROUTE_CASES = [(64, 16, 4, "normal"), (1000, 64, 4, "ties"), (8192, 896, 16, "normal"),
               (257, 896, 16, "ties"), (1, 896, 16, "normal"), (33, 16, 16, "normal"),
               (100, 4096, 32, "normal"), (500, 896, 16, "saturated"), (2048, 448, 8, "zipf"),
               (3, 48, 1, "normal"), (50, 90, 8, "normal"), (700, 1024, 32, "normal"),
               (300, 1024, 32, "ties")]


@pytest.mark.parametrize("T,E,K,kind", ROUTE_CASES)
def test_route_bit_exact(dev, oracle_mod, T, E, K, kind):
    lg = _logits(T, E, kind, seed=T + E + K)
    lg_np = lg.numpy()
    tau_np = oracle_mod.thresholds(lg_np, oracle_mod.fair_share_rank(T, K, E))
    for tau in (tau_np, None):
        idx, gate, sc = lmoe.route(lg.to(dev), None if tau is None else torch.from_numpy(tau).to(dev),
                                   K, want_scores=True)
        r_idx, r_gate, r_sc = oracle_mod.route(lg_np, tau, K)
        assert np.array_equal(sc.cpu().numpy().view(np.int32), r_sc.view(np.int32))
        assert np.array_equal(idx.cpu().numpy(), r_idx)
        assert np.array_equal(gate.cpu().numpy().view(np.int32), r_gate.view(np.int32))


def test_scores_sweep_bit_exact(dev, oracle_mod):
    """The fixed-sequence score over 4.2 M logits spanning [-90, 90], dense near the clamp and
    the subnormal results (z near -88) and near 0: every score bit-equal to the oracle's."""
    parts = [np.linspace(-90.0, 90.0, 2 ** 21, dtype=np.float32),
             np.linspace(-88.5, -86.0, 2 ** 20, dtype=np.float32),
             np.linspace(-1.0, 1.0, 2 ** 20, dtype=np.float32)]
    z = np.concatenate(parts).reshape(4096, 1024)
    _, _, sc = lmoe.route(torch.from_numpy(z).to(dev), None, 1, want_scores=True)
    _, _, r_sc = oracle_mod.route(z, None, 1)
    assert np.array_equal(sc.cpu().numpy().view(np.int32), r_sc.view(np.int32))


THRESH_CASES = [(64, 16, 4, 0), (8192, 896, 16, 0), (32768, 896, 16, 0), (40000, 64, 4, 0),
                (100, 32, 4, 1), (100, 32, 4, 100), (7, 16, 16, 0), (1, 896, 16, 0),
                (3000, 448, 8, 0), (5000, 64, 4, 256), (5000, 64, 4, 257), (8193, 896, 16, 0),
                # the register-resident bit search (T <= 32768, any rank): the extremes of k
                (32768, 16, 16, 32768), (12345, 48, 8, 1), (20000, 32, 4, 4096),
                # the 1024-thread bound-and-select form: ~3600 candidates, four per thread
                (32768, 64, 4, 1000)]


def test_thresholds_many_scores_above_the_bound(dev, oracle_mod):
    """T = 32768 tokens, k = 1000: token t is held by thread t % 1024 of the 1024-thread
    selection.  Lifting the tokens of a few threads far above the rest puts the bound B (the
    k-th largest of the threads' maxima) low in the remaining threads' range.  Column 1 (100
    threads lifted) has ~6600 scores above B, past the 4096 candidates, so the selection falls
    back to the bit search over its registers; column 0 (24 threads) has ~4090, all four
    candidate slots of a thread in use; column 2 (none) ~3800."""
    T, E, k = 32768, 3, 1000
    g = torch.Generator().manual_seed(77)
    lg = torch.randn(T, E, generator=g) * 0.1
    t = torch.arange(T)
    lg[(t % 1024) < 24, 0] += 8.0
    lg[(t % 1024) < 100, 1] += 6.0
    tau = lmoe.thresholds(lg.to(dev), 4, k)
    ref = oracle_mod.thresholds(lg.numpy(), k)
    assert np.array_equal(tau.cpu().numpy().view(np.int32), ref.view(np.int32))


@pytest.mark.parametrize("T,E,K,k_rank", THRESH_CASES)
def test_thresholds_bit_exact(dev, oracle_mod, T, E, K, k_rank):
    for kind in ("normal", "ties", "saturated"):
        lg = _logits(T, E, kind, seed=T * 3 + E)
        tau = lmoe.thresholds(lg.to(dev), K, k_rank)
        k = k_rank if k_rank > 0 else oracle_mod.fair_share_rank(T, K, E)
        ref = oracle_mod.thresholds(lg.numpy(), k)
        assert np.array_equal(tau.cpu().numpy().view(np.int32), ref.view(np.int32)), kind
