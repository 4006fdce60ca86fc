"""The codec-quality study (Fig. 3 and Fig. 4 of "FlashOptim: Optimizers for
Memory Efficient Training", section "实验结果分析") computed on the GPU through
the C ABI, checked against the oracle on the same values, plus the figures'
qualitative claims on the GPU's numbers."""
import numpy as np
import pytest
import torch

import oracle
from quantized_optimizer_state_gb300 import codec_study as cs
from quantized_optimizer_state_gb300 import fo

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fo.lib()
    oracle.build()


def _oracle_stats(theta, rho_bits):
    tp, rho = oracle.split(theta, rho_bits)
    rec = oracle.merge(tp, rho, rho_bits)
    t64 = theta.astype(np.float64)
    rel = np.abs(rec.astype(np.float64) - t64) / t64
    return 100.0 * np.mean(rec.view(np.uint32) == theta.view(np.uint32)), rel.mean(), rel.max()


@pytest.mark.parametrize("e", [-126, -14, 0, 15, 126])
def test_sweep_matches_oracle(e):
    rows = cs.reconstruction_sweep([e], "cuda", stride=4099)
    theta = cs.binade_values(e, "cpu", 4099).numpy()
    for rb in (8, 16):
        ex, mean, mx = _oracle_stats(theta, rb)
        got = rows[0][f"rho{rb}"]
        assert got["exact_percent"] == pytest.approx(ex, rel=0, abs=1e-12)
        assert got["mean_rel"] == pytest.approx(mean, rel=1e-9)
        assert got["max_rel"] == mx


def test_error_is_constant_across_the_fp16_range():
    """Fig. 3: within FP16's range the relative error does not depend on the
    binade (the split is scale-invariant there), for every scheme."""
    rows = cs.reconstruction_sweep([-14, -3, 0, 7, 15], "cuda", stride=97)
    for key in ("rho8", "rho16", "bf16_bf16"):
        first = rows[0][key]
        for r in rows[1:]:
            assert r[key] == first, (key, r["binade"])


def test_page_claims_on_the_gpu_sweep():
    """16-bit rho: 99.92 % bit-exact and mean error below 1e-9; against the
    page's BF16 + BF16 scheme at the same 32 bits, mean and largest errors are
    orders of magnitude smaller."""
    rows = cs.reconstruction_sweep([0], "cuda", stride=1)
    r16, pair = rows[0]["rho16"], rows[0]["bf16_bf16"]
    assert abs(r16["exact_percent"] - 99.92) < 0.005
    assert r16["mean_rel"] < 1e-9
    assert r16["mean_rel"] < pair["mean_rel"] / 1e3
    assert r16["max_rel"] < pair["max_rel"] / 10


def test_nmse_study_matches_oracle():
    m, v = cs.adam_like_state(4096, 3, "cuda")
    for x, kinds in ((m, (fo.FO_STATE_MOMENTUM, fo.FO_STATE_MOMENTUM_LINEAR)),
                     (v, (fo.FO_STATE_VARIANCE, fo.FO_STATE_VARIANCE_LINEAR))):
        xh_host = x.cpu().numpy()
        for kind in kinds:
            gpu = cs.group_nmse(x, cs.quantize_roundtrip(x, kind)).cpu().numpy()
            q, s = oracle.quant_state(xh_host, kind)
            ref = cs.group_nmse(torch.from_numpy(xh_host), torch.from_numpy(oracle.dequant_state(q, s, kind)))
            np.testing.assert_allclose(gpu, ref.numpy(), rtol=1e-6, atol=0)


def test_companding_narrows_the_error_tail():
    """Fig. 4: companding helps the momentum a little and the second moment a
    lot, above all in the tail of the per-group error distribution."""
    r = cs.nmse_study(1 << 14, 5, "cuda")
    m, v = r["momentum"], r["variance"]
    assert m["companded"]["mean"] <= m["linear"]["mean"] * 1.05
    assert v["companded"]["p99"] < v["linear"]["p99"] / 10
    assert v["companded"]["all_zero_groups_percent"] <= v["linear"]["all_zero_groups_percent"]
