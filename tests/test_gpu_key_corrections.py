"""Estimator quality of the four key corrections on the same harness, through
the C ABI: keys quantized into pages, scores read back from the decode
(softmax scale 1, so a score is the estimate of <q, k>).

[Reconstruction] §6: TurboQuant_prod's QJL term makes the inner product
unbiased; §10 / §12.2: EDEN's scale s = ||y||^2 / <y, y_hat> is unbiased as
well, the plain MSE code shrinks it (slope 2/pi at one bit), and the 1-bit
EDEN scalar has a lower variance than a 1-bit QJL sketch; §12 item 2, §13
step 6: TurboVec's length-renormalized correction norm / <y, y_hat> restores
unbiasedness (with the norm stored on its own it is EDEN's scale).  For a query independent of the
key, the code's error r = y - y_hat gives d E<q/||q||, r>^2 = E||r||^2 = D_mse
(the Lloyd-Max unit MSE), and the QJL sketch of r (Gaussian S, d rows) has
variance (pi/2 ||q||^2 ||r||^2 - <q, r>^2) / d, so its distortion is
(pi/2 - 1/d) D_mse -- the figures the pages quote for TurboQuant_prod.

For each (correction, MSE bits) the test measures over 131072 (q, k) pairs of
isotropic bf16 keys (d = 128, dense Pi and FWHT):
    slope = sum est * true / sum true^2      (1 for an unbiased estimator)
    D     = d * mean((est - true)^2 / (||q||^2 ||k||^2))
and prints the table (`pytest -m gpu -s tests/test_gpu_key_corrections.py`); the same for the structured
sketch S = H diag(sigma_S) in place of the Gaussian one.
"""

import numpy as np
import pytest

import synthetic_kv as SK

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

NAMES = {0: "mse", 1: "qjl", 2: "eden", 3: "renorm"}
B, T, HQ, D = 4, 4096, 8, 128


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    from kv_cache_vector_head_gb300 import build

    build.build()
    import kv_cache_vector_head_gb300 as tq

    return tq


def _estimates(tq, w, corr, bits, structured=False):
    """Decode scores (estimates of <q, k>), the exact products and ||q||^2 ||k||^2."""
    L = tq.TQLayer(D, 1, HQ, bits, 2, w.kind, window=0, key_qjl=corr, seed=w.seed, qjl_structured=structured)
    pc = tq.PagedCache(L, B, T)
    kv = SK.keys_values(w)
    k = SK.to_torch(kv["K"], w.dtype).cuda()
    pc.prefill(k, k)
    q = SK.to_torch(kv["q"], w.dtype).cuda()
    ws = torch.empty(tq.decode_workspace_size(L.params, B, T), dtype=torch.uint8, device="cuda")
    out = torch.zeros(B, HQ, D, device="cuda")
    lse = torch.zeros(B, HQ, device="cuda")
    scores = torch.zeros(B, HQ, T, device="cuda")
    tq.decode_attention(L.params, pc.cache, q, 1.0, out, lse, scores, ws, T)
    torch.cuda.synchronize()
    assert tq.check_device_error() == 0
    K = kv["K"][:, :, 0]                      # [B, T, d], float64 of the bf16 values
    Q = kv["q"]                               # [B, Hq, d]
    true = np.einsum("bhd,btd->bht", Q, K)
    qk2 = np.einsum("bh,bt->bht", (Q * Q).sum(-1), (K * K).sum(-1))
    return scores.cpu().numpy().astype(np.float64), true, qk2


@pytest.mark.parametrize("kind", [SK.DENSE, SK.FWHT])
def test_key_correction_estimators(tq, kind):
    w = SK.workload("bulk", batch=B, ctx=T, n_kv_heads=1, n_q_heads=HQ, key_scale="none", value_scale="none",
                    rope=False, kind=kind)
    table = {}
    mse = {bits: tq.build_codebook(D, bits)[2] for bits in (1, 2, 3, 4)}
    for bits in (1, 2, 3, 4):
        for corr in (0, 1, 2, 3):
            est, true, qk2 = _estimates(tq, w, corr, bits)
            slope = float((est * true).sum() / (true * true).sum())
            dist = float(D * np.mean((est - true) ** 2 / qk2))
            table[corr, bits] = (slope, dist)
    print(f"\nkey corrections, d = {D}, {'dense' if kind == SK.DENSE else 'FWHT'}: slope / d * distortion")
    print("bits  " + "  ".join(f"{NAMES[c]:>16}" for c in range(4)))
    for bits in (1, 2, 3, 4):
        print(f"{bits:>4}  " + "  ".join(f"{table[c, bits][0]:7.4f} {table[c, bits][1]:8.5f}" for c in range(4)))
    n = B * HQ * T
    print("Lloyd-Max unit MSE: " + ", ".join(f"{b}: {mse[b]:.5f}" for b in (1, 2, 3, 4)))
    # the structured sketch S = H diag(sigma_S): close to unbiased on the rotated residuals, and its
    # orthogonal rows give a lower distortion than the dense Gaussian sketch
    for bits in (1, 2, 3, 4):
        est, true, qk2 = _estimates(tq, w, 1, bits, structured=True)
        slope = float((est * true).sum() / (true * true).sum())
        dist = float(D * np.mean((est - true) ** 2 / qk2))
        print(f"structured QJL, {bits} bits: slope {slope:.4f}, d * distortion {dist:.5f}")
        tol = 4.0 * np.sqrt(dist / (B * T))
        assert abs(slope - 1.0) < max(tol, 0.01), (bits, slope)
        assert dist < 1.05 * table[1, bits][1], (bits, dist, table[1, bits][1])
    for bits in (1, 2, 3, 4):
        s_mse, d_mse = table[0, bits]
        s_qjl, d_qjl = table[1, bits]
        s_eden, d_eden = table[2, bits]
        s_ren, d_ren = table[3, bits]
        # unbiased estimators: slope 1 within a few standard errors (keys counted once: the
        # eight queries of a key share its code)
        tol = 4.0 * np.sqrt(max(d_qjl, d_eden) / (n / HQ))
        assert abs(s_qjl - 1.0) < max(tol, 0.01), (bits, s_qjl)
        assert abs(s_eden - 1.0) < max(tol, 0.01), (bits, s_eden)
        # TurboVec's correction restores unbiasedness; it stores EDEN's number, so the two agree
        assert abs(s_ren - 1.0) < max(tol, 0.01), (bits, s_ren)
        assert abs(s_ren - s_eden) < 1e-6 and abs(d_ren - d_eden) < 1e-6 * d_eden, (bits, s_ren, s_eden)
        # the plain Lloyd-Max code shrinks the product by 1 - D_mse (centroid condition: E<y, y_hat> =
        # E||y_hat||^2 = 1 - D_mse for a unit y, and the rotation spreads that over every direction)
        assert abs(s_mse - (1.0 - mse[bits])) < max(tol, 0.01), (bits, s_mse, mse[bits])
        # distortion of the plain code D_mse, of the sketch (pi/2 - 1/d) D_mse (sampling: 10 %)
        assert 0.9 < d_mse / mse[bits] < 1.1, (bits, d_mse, mse[bits])
        assert 0.9 < d_qjl / ((np.pi / 2 - 1.0 / D) * mse[bits]) < 1.1, (bits, d_qjl, mse[bits])
    # one MSE bit: the plain code's slope is 2/pi
    assert abs(table[0, 1][0] - 2.0 / np.pi) < 0.02
    # every correction improves with every bit
    for c in range(4):
        assert all(table[c, b][1] > table[c, b + 1][1] for b in (1, 2, 3)), c
