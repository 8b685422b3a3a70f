"""The V^T encoder's division-free quotient, checked on the host.

The encoder codes fl(x / sv) as the sign-flipped E4M3 code of
y = fma(fma(z, sv, x), nr, z), z = fl(x nr), nr = -fl(1/sv) (Markstein's
quotient correction, IBM J. Res. Dev. 34(1), 1990), for scales in
[2^-100, 2^125].  ``tests/v_quotient_check.c`` runs that arithmetic in
IEEE single precision with a correctly rounded fma and compares it with the
oracle's E4M3 code of the quotient fl(x / sv) for every bf16 value up to the
channel maximum: here for every bf16 mantissa of the maximum at exponents
across the range (both end binades included).  The same program with the
argument ``all`` covers every positive finite bf16 maximum (about 1e9 pairs,
a minute and a half).
"""
import os
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("vq") / "v_quotient_check")
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-std=c11",
                    os.path.join(HERE, "v_quotient_check.c"), os.path.join(ROOT, "oracle", "sage_oracle.c"),
                    "-o", exe, "-lm"], check=True)
    return exe


def test_corrected_quotient_codes_equal_the_division(checker):
    out = subprocess.run([checker, "sample"], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout[-2000:]
    pairs = int(out.stdout.split("pairs ")[1].split()[0])
    assert pairs > 30_000_000, out.stdout
    assert "differ 0" in out.stdout, out.stdout
