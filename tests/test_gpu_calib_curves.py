"""GPU parity of the streamed calibration and the distance-preference curves
against the fp64 oracle, through the C ABI.

Streamed calibration: 4096 samples per head fed in uneven chunks (1, 7, 1000,
3088) from the query slice of a fused QKV activation (sample stride (Hq + 2 Hkv)
d), split over two accumulators that are merged, then finalised; compared with
the oracle's one-shot calibration of the same samples at rel 1e-4, and with the
one-shot tri_calibrate_stats.

Curves: pre-RoPE query and key samples of one sequence, centers from
tri_calibrate_stats on each; the center curve and the exact logit curve are
compared with the oracle's (which uses its own fp64 centers and textbook RoPE)
within 1e-3 of the curve's largest magnitude, the correlation within 1e-3.
"""
import numpy as np
import pytest
import torch

import kv_cache_compression_06_b300 as tk
from kv_cache_compression_06_b300 import tri as T
from oracle import tri_oracle as O
from synth import WORKLOADS, Workload, sequence_samples

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def _check_stats(stats, ref, li, rtol=1e-4):
    c, R, m = ref
    gc = stats.center[li].double().cpu().numpy()
    np.testing.assert_allclose(gc[..., 0], c.real, rtol=rtol, atol=1e-5 * np.abs(c).max())
    np.testing.assert_allclose(gc[..., 1], c.imag, rtol=rtol, atol=1e-5 * np.abs(c).max())
    np.testing.assert_allclose(stats.R[li].double().cpu().numpy(), R, rtol=rtol, atol=1e-5)
    np.testing.assert_allclose(stats.mag[li].double().cpu().numpy(), m, rtol=rtol)


@pytest.mark.parametrize("d,dtype,pairing", [(128, torch.bfloat16, "half"), (64, torch.float32, "interleaved"),
                                             (64, torch.bfloat16, "interleaved"), (128, torch.float32, "half")])
def test_streamed_calibration_in_uneven_chunks_matches_one_shot(d, dtype, pairing):
    L, n, Hq, Hkv = 2, 4096, 8, 2
    w = Workload(name=f"calib_stream_{d}", L=L, S=1, Hq=Hq, Hkv=Hkv, d=d, theta=1e6, dtype="bf16", budget=16,
                 offsets=(1,), n_keys=16, mixed_R=True, pairing=pairing)
    qs = [sequence_samples(w, l, n, device=DEV, tag="calib_stream")[0] for l in range(L)]
    q = torch.stack(qs).to(dtype)                                 # [L][n][Hq][d]
    # fused QKV activation [L][n][(Hq + 2 Hkv) d]; the K and V slots hold junk
    qkv = torch.randn((L, n, (Hq + 2 * Hkv) * d), device=DEV).to(dtype)
    qkv[:, :, : Hq * d] = q.reshape(L, n, Hq * d)
    acc_a = T.calib_accumulator(L, Hq, d, DEV)
    acc_b = T.calib_accumulator(L, Hq, d, DEV)
    bounds = np.cumsum([0, 1, 7, 1000, 3088])
    assert bounds[-1] == n
    for c, (i0, i1) in enumerate(zip(bounds[:-1], bounds[1:])):
        view = qkv[:, i0:i1, : Hq * d].unflatten(2, (Hq, d))
        T.tri_calib_accumulate(view, acc_a if c % 2 == 0 else acc_b, pairing=pairing)
    T.tri_calib_accumulate(qkv[:, :0, : Hq * d].unflatten(2, (Hq, d)), acc_b, pairing=pairing)   # n = 0
    T.tri_calib_merge(acc_a, acc_b)
    stats = T.tri_calib_finalize(acc_a)
    one_shot = tk.tri_calibrate_stats(q.contiguous(), pairing=pairing)
    torch.cuda.synchronize()
    assert acc_a[..., 6].min().item() == n and acc_a[..., 6].max().item() == n
    for li in range(L):
        _check_stats(stats, O.calibrate(q[li].double().cpu().numpy(), pairing), li)
    for a, b in ((stats.center, one_shot.center), (stats.R, one_shot.R), (stats.mag, one_shot.mag)):
        torch.testing.assert_close(a, b, rtol=1e-5, atol=1e-6)


def test_streamed_calibration_reset_and_zero_count_bands():
    """A reset accumulator finalises to zeros (no samples); all-zero samples
    count toward the means but not toward R."""
    L, H, d = 1, 2, 64
    acc = T.calib_accumulator(L, H, d, DEV)
    st = T.tri_calib_finalize(acc)
    torch.cuda.synchronize()
    assert torch.count_nonzero(st.center) == 0 and torch.count_nonzero(st.R) == 0 and torch.count_nonzero(st.mag) == 0
    q = torch.zeros((L, 10, H, d), device=DEV)
    q[0, :4, 0, 0] = 1.0                 # head 0, band 0 (rotate-half): 4 unit samples, 6 zero samples
    T.tri_calib_accumulate(q, acc)
    st = T.tri_calib_finalize(acc)
    torch.cuda.synchronize()
    assert abs(st.center[0, 0, 0, 0].item() - 0.4) < 1e-7 and abs(st.mag[0, 0, 0].item() - 0.4) < 1e-7
    assert abs(st.R[0, 0, 0].item() - 1.0) < 1e-7
    assert st.R[0, 1].abs().max().item() == 0.0


CURVE_CASES = [
    # (Hq, Hkv, d, dtype, pairing, n, n_delta)
    (8, 2, 128, torch.bfloat16, "half", 1024, 256),
    (4, 4, 64, torch.float32, "interleaved", 600, 600),     # G = 1, every distance up to n - 1
    (8, 1, 128, torch.float32, "half", 333, 100),          # ragged tails of both tilings
]


@pytest.mark.parametrize("case", CURVE_CASES, ids=[f"g{c[0] // c[1]}_d{c[2]}_{c[4]}_n{c[5]}" for c in CURVE_CASES])
def test_distance_curves_match_oracle(case):
    Hq, Hkv, d, dtype, pairing, n, nd = case
    w = Workload(name=f"curves_{Hq}_{Hkv}_{d}", L=1, S=1, Hq=Hq, Hkv=Hkv, d=d, theta=1e6, dtype="bf16",
                 budget=16, offsets=(1,), n_keys=16, mixed_R=True, pairing=pairing)
    q, k, _ = sequence_samples(w, 0, n, device=DEV, tag="curves_gpu")
    q, k = q.to(dtype), k.to(dtype)
    sq = tk.tri_calibrate_stats(q[None].contiguous(), pairing=pairing)
    sk = tk.tri_calibrate_stats(k[None].contiguous(), pairing=pairing)
    cc, lc, corr = T.tri_distance_curves(sq.center, sk.center, q[None], k[None], w.theta, nd, pairing=pairing)
    torch.cuda.synchronize()
    qn, kn = q.double().cpu().numpy(), k.double().cpu().numpy()
    cq, _, _ = O.calibrate(qn, pairing)
    ck, _, _ = O.calibrate(kn, pairing)
    G = Hq // Hkv
    for h in range(Hq):
        c_ref = O.center_curve(cq[h], ck[h // G], d, w.theta, nd)
        e_ref = O.logit_curve(qn[:, h], kn[:, h // G], w.theta, nd, pairing)
        c_gpu = cc[0, h].double().cpu().numpy()
        e_gpu = lc[0, h].double().cpu().numpy()
        assert np.abs(c_gpu - c_ref).max() <= 1e-3 * np.abs(c_ref).max(), h
        assert np.abs(e_gpu - e_ref).max() <= 1e-3 * np.abs(e_ref).max(), h
        assert abs(corr[0, h].item() - O.pearson(c_ref, e_ref)) <= 1e-3, h


def test_center_curve_only():
    """logit_curve and corr omitted: the sequences are not read."""
    F = 64
    cq = torch.randn((2, 4, F, 2), device=DEV)
    ck = torch.randn((2, 2, F, 2), device=DEV)
    cc, lc, corr = T.tri_distance_curves(cq, ck, None, None, 1e6, 50)
    torch.cuda.synchronize()
    assert lc is None and corr is None
    for l in range(2):
        for h in range(4):
            a = cq[l, h].double().cpu().numpy()
            b = ck[l, h // 2].double().cpu().numpy()
            ref = O.center_curve(a[:, 0] + 1j * a[:, 1], b[:, 0] + 1j * b[:, 1], 2 * F, 1e6, 50)
            assert np.abs(cc[l, h].double().cpu().numpy() - ref).max() <= 1e-4 * np.abs(ref).max()
