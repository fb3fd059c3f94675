"""Plant plausible mistakes in a private copy of the oracle's C source and check that
the pins catch every one of them (a pin that passes a broken oracle pins nothing)."""
import importlib.util
import os
import shutil

import pytest

import oracle
import pins

# (description, text in attn_oracle.c, replacement)
MUTANTS = [
    ("softmax scale dropped", "s[j] = scale * acc;", "s[j] = acc;"),
    ("no division by l", "double p = exp(s[j] - m) / l;", "double p = exp(s[j] - m);"),
    ("LSE without the max", "lse[bh * nout + r] = m + log(l);", "lse[bh * nout + r] = log(l);"),
    ("l without the max shift", "l += exp(s[j] - m);", "l += exp(s[j]);"),
    ("causal mask one key late", "return causal ? (i + (Nk - Nq) + 1) : Nk;",
     "return causal ? (i + (Nk - Nq) + 2 > Nk ? Nk : i + (Nk - Nq) + 2) : Nk;"),
    ("V rows reversed", "const double *vj = vh + j * d;", "const double *vj = vh + (nk - 1 - j) * d;"),
    ("dP with transposed indices", "dp += doh[i * d + t] * vh[j * d + t];",
     "dp += doh[j * d + t] * vh[i * d + t];"),
    ("dS sign flipped", "double ds = p * (dp - c[i]);", "double ds = p * (c[i] - dp);"),
    ("dS without the row term", "double ds = p * (dp - c[i]);", "double ds = p * dp;"),
    ("row term without P", "acc += p * dp;", "acc += dp;"),
    ("dV from Q instead of dO", "gv[t] += p * doh[i * d + t];", "gv[t] += p * qh[i * d + t];"),
    ("dK without scale", "gk[t] += scale * ds * qh[i * d + t];", "gk[t] += ds * qh[i * d + t];"),
    ("dQ from V instead of K", "g[t] += scale * ds * kh[j * d + t];", "g[t] += scale * ds * vh[j * d + t];"),
    ("causal backward sees every query", "int64_t i0 = causal ? j - (Nk - N) : 0;", "int64_t i0 = 0;"),
    ("e4m3 exponent bias 8", "mag = ldexp(1.0 + (double)man / 8.0, e - 7);",
     "mag = ldexp(1.0 + (double)man / 8.0, e - 8);"),
    ("e4m3 mantissa in sixteenths", "mag = ldexp(1.0 + (double)man / 8.0, e - 7);",
     "mag = ldexp(1.0 + (double)man / 16.0, e - 7);"),
    ("e4m3 subnormals at 2^-7", "mag = ldexp((double)man / 8.0, -6);", "mag = ldexp((double)man / 8.0, -7);"),
    ("e4m3 sign dropped", "return sgn ? -mag : mag;", "return mag;"),
    ("block scale indexed by row modulo", "scales[bh * nblk + n / block_rows]", "scales[bh * nblk + n % nblk]"),
    ("one scale per head", "scales[bh * nblk + n / block_rows]", "scales[bh * nblk]"),
    ("rectangular causal aligned to the first key", "return causal ? (i + (Nk - Nq) + 1) : Nk;",
     "return causal ? (i + 1) : Nk;"),
    ("rectangular causal backward without the offset", "int64_t i0 = causal ? j - (Nk - N) : 0;",
     "int64_t i0 = causal ? j : 0;"),
    ("philox multiplier off by two", "(uint64_t)0xD2511F53u * c0", "(uint64_t)0xD2511F55u * c0"),
    ("philox key bump dropped", "k1 += 0xBB67AE85u;", ""),
    ("dropout without the rescale", "return byte >= (uint32_t)t ? 256.0 / (256.0 - t) : 0.0;",
     "return byte >= (uint32_t)t ? 1.0 : 0.0;"),
    ("dropout bytes big-endian", "(w[b / 4] >> (8 * (b % 4)))", "(w[b / 4] >> (24 - 8 * (b % 4)))"),
    ("dropout counter fields swapped", "{(uint32_t)(j / 16), (uint32_t)i, (uint32_t)bh, 0u}",
     "{(uint32_t)(i / 16), (uint32_t)j, (uint32_t)bh, 0u}"),
    ("dropout row term without the keep factor", "acc += p * z * dpt;", "acc += p * dpt;"),
    ("dropout dV without the keep factor", "gv[x] += p * z * doh[i * d + x];", "gv[x] += p * doh[i * d + x];"),
    ("dropout dS without the keep factor", "double ds = p * (z * dpt - c[i]);", "double ds = p * (dpt - c[i]);"),
    ("dropout forward ignores the head offset", "double pz = exp(s[j] - m) / l * oracle_dropout_factor(bh0 + bh,",
     "double pz = exp(s[j] - m) / l * oracle_dropout_factor(bh,"),
    ("dropout backward ignores the head offset", "double z = oracle_dropout_factor(bh0 + bh, i, j, t, seed_lo, seed_hi);",
     "double z = oracle_dropout_factor(bh, i, j, t, seed_lo, seed_hi);"),
]


@pytest.mark.parametrize("desc,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, desc, old, new):
    src = open(oracle.SOURCE).read()
    assert old in src, f"mutation site for '{desc}' not found in the oracle source"
    mutated = src.replace(old, new)
    c_path = os.path.join(tmp_path, "mutant.c")
    open(c_path, "w").write(mutated)
    lib = oracle.build(force=True, src=c_path, out=os.path.join(tmp_path, "libmutant.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, RuntimeError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the mutant '{desc}'"


# Mistakes in the Python composition of the packed-batch oracle (oracle/__init__.py):
# (description, text, replacement), applied to a private copy of the module.
PY_MUTANTS = [
    ("packed dK taken from dV", "gq.transpose(1, 0, 2), gk.transpose(1, 0, 2), gv.transpose(1, 0, 2)",
     "gq.transpose(1, 0, 2), gv.transpose(1, 0, 2), gv.transpose(1, 0, 2)"),
    ("packed dK scattered into the query slice", "dq[qs], dk[ks], dv[ks] =", "dq[qs], dk[qs], dv[ks] ="),
    ("packed backward skips sequences with Nk != Nq", "if nq == 0 or self._degenerate(nq, nk, causal):",
     "if nq == 0 or nq != nk or self._degenerate(nq, nk, causal):"),
    ("packed backward ignores the causal flag", "t(do, qs), causal, scale)", "t(do, qs), False, scale)"),
    ("packed forward: degenerate rows get lse 0", "lse[:, qs] = -np.inf", "lse[:, qs] = 0.0"),
]


@pytest.mark.parametrize("desc,old,new", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_pins_catch_python_mutant(tmp_path, desc, old, new):
    src = open(os.path.join(os.path.dirname(oracle.SOURCE), "__init__.py")).read()
    assert old in src, f"mutation site for '{desc}' not found in the oracle module"
    pkg = os.path.join(tmp_path, "oracle_mutant")
    os.makedirs(pkg)
    open(os.path.join(pkg, "__init__.py"), "w").write(src.replace(old, new))
    shutil.copy(oracle.SOURCE, os.path.join(pkg, "attn_oracle.c"))
    spec = importlib.util.spec_from_file_location("oracle_mutant_%d" % abs(hash(desc)), os.path.join(pkg, "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    orc = mod.Oracle(oracle.default().path)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, RuntimeError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the mutant '{desc}'"
