"""The pins are strong enough: each plausible mistake planted in a copy of the
oracle (a dropped term, a wrong sign or index, a swapped operand, an
off-by-one mask) makes at least one pin fail.

The mistakes are planted on the CPU, in a temporary copy of the oracle's C
source compiled with gcc; the committed oracle is untouched.
"""
import math
import os
import subprocess

import numpy as np
import pytest

import oracle
from test_oracle_pins import brute_force, torch_reference

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "causal_off_by_one": ("if (causal && j > i) return 0;", "if (causal && j >= i) return 0;"),
    "window_off_by_one": ("if (wl >= 0 && j < i - wl) return 0;",
                          "if (wl >= 0 && j <= i - wl) return 0;"),
    "scale_dropped": ("S[r * Sk + j] = scale * dot;", "S[r * Sk + j] = dot;"),
    "wrong_key_index": ("const double *kj = kbh + j * D;",
                        "const double *kj = kbh + (Sk - 1 - j) * D;"),
    "max_sign": ("const double e = exp(S[r * Sk + j] - m);",
                 "const double e = exp(S[r * Sk + j] + m);"),
    "no_normalisation": ("for (long j = 0; j < Sk; ++j) P[r * Sk + j] /= sum;", ""),
    "lse_drops_max": ("lrow_base[lidx[r]] = m + log(sum);", "lrow_base[lidx[r]] = log(sum);"),
    "v_is_k": ("const double *vj = vbh + j * D;", "const double *vj = kbh + j * D;"),
    "transposed_q": ("const double *qi = qbh + i * D;", "const double *qi = qbh + i;"),
    "bf16_widening": ("uint32_t u = ((uint32_t)h) << 16;", "uint32_t u = ((uint32_t)h) << 15;"),
}

# mistakes planted in the backward pass
BWD_MUTANTS = {
    "delta_sign": ("dS[i * Sk + j] = P[i * Sk + j] * (dp - dl);", "dS[i * Sk + j] = P[i * Sk + j] * (dp + dl);"),
    "dq_no_scale": ("dq[i * D + d] = jb->scale * a;", "dq[i * D + d] = a;"),
    "dk_uses_k": ("a += dS[i * Sk + j] * Q[i * D + d];", "a += dS[i * Sk + j] * K[i * D + d];"),
    "dv_transposed_p": ("b += P[i * Sk + j] * G[i * D + d];", "b += P[j * Sk + i] * G[i * D + d];"),
    "delta_uses_v": ("for (long d = 0; d < D; ++d) dl += G[i * D + d] * O[i * D + d];",
                     "for (long d = 0; d < D; ++d) dl += G[i * D + d] * V[i * D + d];"),
}


def _pins_pass(lib) -> bool:
    """A small battery of the pins; True only if every one holds."""
    rng = np.random.default_rng(2024)
    try:
        for causal, window in [(False, (-1, -1)), (True, (-1, -1)), (True, (1, -1))]:
            q, k, v = (rng.standard_normal((1, 2, 4, 3)) for _ in range(3))
            o, lse = oracle.attn_fwd(q, k, v, 0.7, causal, window, lib=lib)
            ob, lb = brute_force(q, k, v, 0.7, causal, *window)
            if not (np.allclose(o, ob, rtol=0, atol=1e-12)
                    and np.allclose(lse, lb, rtol=0, atol=1e-12)):
                return False
        q, k, v = (rng.standard_normal((1, 1, 40, 16)) for _ in range(3))
        o, lse = oracle.attn_fwd(q, k, v, 0.25, True, lib=lib)
        ot, lt = torch_reference(q, k, v, 0.25, True)
        if not (np.allclose(o, ot, atol=1e-12) and np.allclose(lse, lt, atol=1e-12)):
            return False
        # bf16 front end must be the exact widening
        # moderate magnitudes: sign | exponent 120..130 | random mantissa
        expo = rng.integers(120, 131, size=(1, 1, 8, 4))
        bits = ((rng.integers(0, 2, size=expo.shape) << 15) | (expo << 7)
                | rng.integers(0, 128, size=expo.shape)).astype(np.uint16)
        wide = oracle.bf16_bits_to_f64(bits)
        o1, l1 = oracle.attn_fwd(bits, bits, bits, 0.5, False, lib=lib)
        o2, l2 = oracle.attn_fwd(wide, wide, wide, 0.5, False, lib=lib)
        if not (np.array_equal(o1, o2) and np.array_equal(l1, l2)):
            return False
    except oracle.OracleError:
        return False
    return bool(math.isfinite(float(lse.sum())))


def test_unmutated_oracle_passes_battery(oracle_lib):
    assert _pins_pass(oracle_lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(before) == 1, f"mutation anchor for {name} not unique"
    src = tmp_path / f"mutant_{name}.c"
    src.write_text(text.replace(before, after))
    out = str(tmp_path / f"libmutant_{name}.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", out,
                    str(src), "-lm"], check=True)
    lib = oracle.load(out)
    assert not _pins_pass(lib), f"planted mistake {name} was not caught by the pins"


def _bwd_pins_pass(lib) -> bool:
    """Finite differences of the unmutated forward and torch autograd."""
    from test_oracle_bwd_pins import _loss
    rng = np.random.default_rng(5)
    q, k, v, g = (rng.standard_normal((1, 1, 4, 3)) for _ in range(4))
    try:
        dq, dk, dv = oracle.attn_bwd(q, k, v, g, 0.8, True, lib=lib)
    except oracle.OracleError:
        return False
    good = oracle.load()
    h = 1e-5
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            a = {"q": q, "k": k, "v": v}
            b = dict(a)
            a[name], b[name] = xp, xm
            num = (_loss(a["q"], a["k"], a["v"], g, 0.8, True, (-1, -1), good)
                   - _loss(b["q"], b["k"], b["v"], g, 0.8, True, (-1, -1), good)) / (2 * h)
            if not abs(num - grad[idx]) <= 1e-8:
                return False
    return True


def test_unmutated_backward_passes_battery(oracle_lib):
    assert _bwd_pins_pass(oracle_lib)


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_planted_backward_mistake_is_caught(name, tmp_path):
    before, after = BWD_MUTANTS[name]
    text = open(SRC).read()
    assert text.count(before) == 1, f"mutation anchor for {name} not unique"
    src = tmp_path / f"mutant_{name}.c"
    src.write_text(text.replace(before, after))
    out = str(tmp_path / f"libmutant_{name}.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", out,
                    str(src), "-lm"], check=True)
    assert not _bwd_pins_pass(oracle.load(out)), f"planted mistake {name} was not caught"
