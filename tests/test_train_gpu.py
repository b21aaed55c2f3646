"""Training-time expanded projection on the GPU against the fp64 oracle: K_h = X (W_shared +
U_h B_h^T) forward, and the chain-rule gradients dX, dW_shared, dU_h, dB_h ("Low-Rank Key Value
Attention", frame "Training learns the base and residuals together").  The GPU rounds S, R and
the backward's [G | dR] to bf16 between its tensor-core products (fp32 accumulation), so results
are compared at the decode tolerance (relative L2 5e-3, max abs 2e-2 scaled to the output size)."""
import numpy as np
import pytest
import torch

import lrkv_synth as S
import oracle
from cases import f64
from gpu_util import dev_bf16, errors, host_f64

pytestmark = pytest.mark.gpu

from compressed_kv_cache_lrkv_gb300 import binding as b  # noqa: E402


def _check(got, ref, what, rel_tol=5e-3):
    rel, mx = errors(got, ref)
    scale = float(np.max(np.abs(ref))) if ref.size else 1.0
    assert np.all(np.isfinite(got)), what
    assert rel <= rel_tol and mx <= 2e-2 * max(scale, 1.0), f"{what}: rel_l2={rel:.3e} max_abs={mx:.3e} scale={scale:.3e}"


def run_train(n, d, d_h, H, r, seed):
    X = S.gaussian_bf16(seed, "X", (n, d))
    Ws = S.gaussian_bf16(seed, "Ws", (d, d_h), d ** -0.5)
    U = S.gaussian_bf16(seed, "U", (H, d, r), d ** -0.5)
    Bm = S.gaussian_bf16(seed, "B", (H, d_h, r), r ** -0.5)
    dK = S.gaussian_bf16(seed, "dK", (n, H, d_h))
    dims = b.make_dims(H, d_h, r, d)
    tX, tWs, tU, tB, tdK = (dev_bf16(a) for a in (X, Ws, U, Bm, dK))
    Wt = b.pack_side_t(tWs, tU)
    Ncat = d_h + H * r
    Y = torch.empty(n, Ncat, dtype=torch.bfloat16, device="cuda")
    K = torch.empty(n, H, d_h, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.lrkv_train_forward(dims, tX, Wt, tB, Y, K, status=st)
    dX = torch.empty(n, d, dtype=torch.bfloat16, device="cuda")
    dWt = torch.empty(Ncat, d, dtype=torch.bfloat16, device="cuda")
    dB = torch.empty(H, d_h, r, dtype=torch.bfloat16, device="cuda")
    ws = b.alloc_workspace(b.train_workspace_bytes(dims, n))
    b.lrkv_train_backward(dims, tX, Wt, tB, Y, tdK, dX, dWt, dB, ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return (X, Ws, U, Bm, dK), (host_f64(K), host_f64(dX), host_f64(dWt), host_f64(dB), host_f64(Y))


SHAPES = [
    # n, d, d_h, H, r
    (256, 512, 64, 8, 8),
    (300, 512, 64, 8, 16),       # ragged token count
    (1000, 1024, 128, 4, 32),
    (512, 4096, 128, 32, 16),    # the 6.3B head shape
    (77, 264, 128, 3, 16),       # d not a multiple of 64, few tokens
]


@pytest.mark.parametrize("n,d,d_h,H,r", SHAPES, ids=[f"n{s[0]}_d{s[1]}_dh{s[2]}_H{s[3]}_r{s[4]}" for s in SHAPES])
def test_train_forward_backward_match_oracle(n, d, d_h, H, r):
    (X, Ws, U, Bm, dK), (K, dX, dWt, dB, Y) = run_train(n, d, d_h, H, r, 600 + n + H)
    o = oracle.get()
    _check(K, o.train_forward(X, Ws, U, Bm), "K")
    rdX, rdWs, rdU, rdB = o.train_backward(X, Ws, U, Bm, dK)
    _check(dX, rdX, "dX")
    _check(dWt[:d_h], rdWs.T, "dW_shared^T")
    _check(dWt[d_h:].reshape(H, r, d), np.transpose(rdU, (0, 2, 1)), "dU^T")
    _check(dB, rdB, "dB")
    # Y holds the factored features [S | R] = X [W_shared | U_1 .. U_H] rounded to bf16
    ref_Y = f64(X) @ np.concatenate([f64(Ws), np.transpose(f64(U), (1, 0, 2)).reshape(d, H * r)], axis=1)
    _check(Y, ref_Y, "Y")


def test_train_zero_tokens_is_noop():
    dims = b.make_dims(8, 64, 8, 512)
    z = torch.empty(0, 512, dtype=torch.bfloat16, device="cuda")
    b.lrkv_train_forward(dims, z, z, z, z, z)


def test_train_full_size_sampled():
    """The timed training workload's launch configuration (8192 tokens, d=4096, H=32, d_h=128, r=16:
    every GEMM loops over several tiles per CTA, so both accumulator buffers, the staging boxes and
    the ring phases wrap), checked on outputs the oracle computes from a slice of the inputs:
    K and dX rows from their own tokens, dW_T columns from their own feature columns of X (G and
    dR do not depend on X), dB of two heads from those heads' factors and gradients."""
    wl = S.WORKLOADS["train"]
    n, d, d_h, H, r = wl.B * wl.L, wl.d, wl.d_h, wl.H, wl.r
    (X, Ws, U, Bm, dK), (K, dX, dWt, dB, Y) = run_train(n, d, d_h, H, r, wl.seed)
    o = oracle.get()
    rows = np.unique(np.concatenate([np.arange(0, 8), np.arange(n - 8, n),
                                     np.random.default_rng(wl.seed).choice(n, 48, replace=False)]))
    _check(K[rows], o.train_forward(X[rows], Ws, U, Bm), "K rows")
    rdX, _, _, _ = o.train_backward(X[rows], Ws, U, Bm, dK[rows])
    _check(dX[rows], rdX, "dX rows")
    cols = np.unique(np.concatenate([np.arange(0, 4), np.arange(d - 4, d),
                                     np.random.default_rng(wl.seed + 1).choice(d, 8, replace=False)]))
    _, rdWs, rdU, _ = o.train_backward(np.ascontiguousarray(X[:, cols]), np.ascontiguousarray(Ws[cols]),
                                       np.ascontiguousarray(U[:, cols]), Bm, dK)
    _check(dWt[:d_h][:, cols], rdWs.T, "dW_shared^T columns")
    _check(dWt[d_h:].reshape(H, r, d)[:, :, cols], np.transpose(rdU, (0, 2, 1)), "dU^T columns")
    hs = np.array([0, H - 1])
    _, _, _, rdB = o.train_backward(X, Ws, np.ascontiguousarray(U[hs]), np.ascontiguousarray(Bm[hs]),
                                    np.ascontiguousarray(dK[:, hs]))
    _check(dB[hs], rdB, "dB heads")
