"""The oracle's pins must catch plausible mistakes (not gpu).

Each case plants one mistake in a temporary copy of oracle.c (on the CPU, in a
scratch directory), rebuilds it there and runs the oracle pin tests against
the copy; the run must fail.  Mistakes: a wrong twist root, a missing output
bit reversal, a '+' for the negacyclic '-', a lost automorphism sign, a
Garner radix error, a non-minimal root, a missing 1/n, swapped key
components, a wrong tensor cross term, a wrong prime step, a dropped
Miller-Rabin round, two ModDown rounding mistakes, two approximate basis
conversion mistakes, two hoisted key-switch mistakes, an inverse twist by
the forward root, a cyclic transform by psi instead of psi^2, a wrong
extension radix, a ModDown by P instead of P^-1, a digit width rounded down
and an NTT-domain automorphism composed in the wrong order.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "twist_uses_inverse_root": (
        "a[j] = mulmod(a[j] % q, pw, q); pw = mulmod(pw, psi, q);",
        "a[j] = mulmod(a[j] % q, pw, q); pw = mulmod(pw, invmod(psi, q), q);"),
    "no_output_bit_reversal": (
        "    /* A[k] is the value at psi^(2k+1); the definition stores it at brv(k) */\n"
        "    bit_reverse_permute(a, log_n);\n", ""),
    "negacyclic_wrap_added": (
        "else c[i + j - n] = submod(c[i + j - n], p, q);",
        "else c[i + j - n] = addmod(c[i + j - n], p, q);"),
    "automorph_sign_lost": (
        "else out[s - n] = (q - a[t] % q) % q;",
        "else out[s - n] = a[t] % q;"),
    "garner_radix_wrong": (
        "radix = mulmod(radix, d[k] % qi, qi);",
        "radix = mulmod(radix, d[k] % qi, qi); if (k == 1) radix = mulmod(radix, 2, qi);"),
    "psi_not_smallest": (
        "if (cur < best) best = cur;",
        "if (cur > best) best = cur;"),
    "missing_n_inverse": (
        "uint64_t n_inv = invmod(n % q, q), pw = n_inv;",
        "uint64_t pw = 1;"),
    "key_components_swapped": (
        "uint64_t kv = keys[(((uint64_t)j * 2 + c) * LK + l) * n + i];",
        "uint64_t kv = keys[(((uint64_t)j * 2 + (1 - c)) * LK + l) * n + i];"),
    "tensor_cross_term_wrong": (
        "d1[o] = addmod(mulmod(a0[o], b1[o], ql), mulmod(a1[o], b0[o], ql), ql);",
        "d1[o] = addmod(mulmod(a0[o], b0[o], ql), mulmod(a1[o], b1[o], ql), ql);"),
    "prime_scan_skips": (
        "        c -= m;\n    }\n    return found;",
        "        c -= 2 * m;\n    }\n    return found;"),
    "moddown_rounding_sign": (
        "uint64_t num = submod(addmod(x[l] % q, h, q), c, q);",
        "uint64_t num = submod(submod(x[l] % q, h, q), c, q);"),
    "moddown_rounding_missing_on_p": (
        "uint64_t h = nearest ? (P[k] - 1) / 2 : 0;",
        "uint64_t h = 0;"),
    "fast_bconv_missing_qhat_inverse": (
        "for (int j = 0; j < S; j++) y[j] = mulmod(x[j] % src[j], qinv[j], src[j]);",
        "for (int j = 0; j < S; j++) y[j] = x[j] % src[j];"),
    "fast_bconv_qhat_keeps_own_prime": (
        "if (i != j) h = mulmod(h, src[i] % p, p);",
        "h = mulmod(h, src[i] % p, p);"),
    "hoisted_skips_automorphism": (
        "oracle_automorph_batch(ext, rot, log_n, LK, batch * dnum, qp, psi_qp, ks[r], 1, threads);",
        "memcpy(rot, ext, rows * sizeof(uint64_t));"),
    "hoisted_automorphism_in_wrong_domain": (
        "oracle_automorph_batch(ext, rot, log_n, LK, batch * dnum, qp, psi_qp, ks[r], 1, threads);",
        "oracle_automorph_batch(ext, rot, log_n, LK, batch * dnum, qp, psi_qp, ks[r], 0, threads);"),
    "intt_twist_uses_forward_root": (
        "for (uint64_t j = 0; j < n; j++) { a[j] = mulmod(a[j], pw, q); pw = mulmod(pw, psi_inv, q); }",
        "for (uint64_t j = 0; j < n; j++) { a[j] = mulmod(a[j], pw, q); pw = mulmod(pw, psi, q); }"),
    "ntt_cyclic_root_not_squared": (
        "cyclic_dft(a, log_n, q, mulmod(psi, psi, q));",
        "cyclic_dft(a, log_n, q, psi);"),
    "extension_radix_wrong": (
        "        acc = addmod(acc, mulmod(v[i] % p, radix, p), p);\n        radix = mulmod(radix, d[i] % p, p);",
        "        acc = addmod(acc, mulmod(v[i] % p, radix, p), p);\n        radix = mulmod(radix, d[i] % p, p);"
        " if (i == 0) radix = addmod(radix, 1, p);"),
    "moddown_multiplies_by_P": (
        "out[l] = mulmod(num, invmod(Pm, q), q);",
        "out[l] = mulmod(num, Pm, q);"),
    "digit_width_rounded_down": (
        "    int alpha = (L + dnum - 1) / dnum;\n    *lo = j * alpha;",
        "    int alpha = L / dnum;\n    *lo = j * alpha;"),
    "automorph_ntt_domain_composed_backwards": (
        "    oracle_intt(tmp, log_n, q, psi);\n    oracle_automorph_coeff(tmp, out, log_n, q, k);\n"
        "    oracle_ntt(out, log_n, q, psi);",
        "    oracle_ntt(tmp, log_n, q, psi);\n    oracle_automorph_coeff(tmp, out, log_n, q, k);\n"
        "    oracle_intt(out, log_n, q, psi);"),
    "miller_rabin_one_round": (
        "    for (int i = 0; i < 12; i++) {\n        uint64_t x = powmod(small[i], d, n);",
        "    for (int i = 0; i < 1; i++) {\n        uint64_t x = powmod(small[i], d, n);"),
}

PIN_FILES = ["test_oracle_primes_psi.py", "test_oracle_ntt.py", "test_oracle_automorph.py",
             "test_oracle_keyswitch.py", "test_oracle_moddown.py", "test_oracle_bconv.py"]


@pytest.fixture(scope="module")
def source():
    with open(os.path.join(ROOT, "oracle", "oracle.c")) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    work = tmp_path / "w"
    shutil.copytree(os.path.join(ROOT, "oracle"), work / "oracle",
                    ignore=shutil.ignore_patterns("*.so", "*.tmp*", "__pycache__"))
    shutil.copytree(os.path.join(ROOT, "ntt_arithmetic_gb300"), work / "ntt_arithmetic_gb300",
                    ignore=shutil.ignore_patterns("*.so", "__pycache__", "_build", "csrc"))
    (work / "tests").mkdir()
    for f in PIN_FILES + ["conftest.py"]:
        shutil.copy(os.path.join(ROOT, "tests", f), work / "tests" / f)
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), work / "tests" / "golden")
    (work / "oracle" / "oracle.c").write_text(source.replace(old, new))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider",
                        "tests"], cwd=work, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout or "error" in r.stdout.lower()
