"""The kernels divide every value of a block by that block's scale with one correctly rounded
reciprocal and Markstein's remainder correction (P. Markstein, IBM J. Res. Dev. 34(1), 1990),
run on negated values so that signed zeros keep their sign.  The definition asks for IEEE
fp32 division ("A Fused Hadamard + NVFP4 Quantization Kernel in Triton", §1 table and §2
kernel: y / s_f).  This checks on the host CPU that the method equals IEEE division over
5.2e9 operand pairs (all divisor mantissas; all dividend mantissas for 600 divisors)."""
import os
import platform
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))


def test_markstein_equals_ieee_division(tmp_path):
    exe = tmp_path / "division_method"
    # fmaf is correctly rounded with or without a hardware FMA; -mfma only makes it fast on x86.
    extra = ["-mfma"] if platform.machine() == "x86_64" else []
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", *extra, "-o", str(exe),
                    os.path.join(HERE, "csrc", "division_method.c"), "-lm"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout
    assert "mismatches 0" in out.stdout, out.stdout
