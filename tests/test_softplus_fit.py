"""The scan kernel's softplus polynomial against its fitting script: the
coefficients in csrc/scan.cu are the ones hybrid_attention_ssm_fwd_b300/
fit_softplus.py produces (up to the fit's convergence noise), and e * q(e),
evaluated in float32 as the kernel does, stays within 4e-7 relative of
log1p(e) on (0, 1] -- so softplus(v) = max(v, 0) + e q(e), e = exp(-|v|),
keeps that bound for every v."""
import os
import re

import numpy as np

from hybrid_attention_ssm_fwd_b300 import fit_softplus as fs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def kernel_coefficients():
    src = open(os.path.join(ROOT, "hybrid_attention_ssm_fwd_b300", "csrc", "scan.cu")).read()
    body = src[src.index("HY_DEV float softplus_scan(float v)"):]
    body = body[: body.index("return fmaxf")]
    first = re.search(r"float q = (-?[0-9.e-]+)f;", body).group(1)
    rest = re.findall(r"q = fmaf\(q, e, (-?[0-9.e-]+)f\);", body)
    return np.array([float(first)] + [float(v) for v in rest], np.float32)


def test_kernel_coefficients_are_the_fit():
    ck = kernel_coefficients()
    cf = fs.fit()
    assert len(ck) == fs.DEGREE + 1
    np.testing.assert_allclose(ck, cf, atol=2e-6, rtol=0)


def test_kernel_polynomial_error_bound():
    assert fs.max_rel_error(kernel_coefficients()) < 4e-7
    assert fs.max_rel_error(fs.fit()) < 4e-7


def test_target_limit_and_values():
    np.testing.assert_allclose(fs.target(np.array([0.0, 1.0])), [1.0, np.log(2.0)], rtol=1e-15)
