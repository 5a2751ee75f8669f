"""Mutation check of the oracle's pins:  python tests/oracle_mutations.py [name ...]

Each entry below plants one plausible mistake in the oracle (a dropped term, a wrong sign,
index, divisor or rounding, a swapped or transposed operand), by replacing one exact
substring of oracle/qs_oracle.c (or of the named oracle file) that must occur once.  The mistake goes into a copy of
oracle/, qs_inputs/ and tests/ in a temporary directory, never into the repository.  Then
the oracle pins run there (the CPU tests test_oracle_*.py).  Every mutation must make a pin
fail; one that does not is reported as SURVIVED, and the script exits non-zero.  Every
planted index stays inside its buffer, so a mutant cannot crash the test process.  Not
collected by pytest: it takes a few seconds per mutation.
"""
import os
import shutil
import subprocess
import sys
import tempfile

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE = None  # the temporary mirror, set in main()

M = [
    ("q2k unpack shift", "(blk[16 + 32 * h + l] >> (2 * j)) & 3)", "(blk[16 + 32 * h + l] >> (2 * j + 1)) & 3)"),
    ("q2k unpack halves swapped", "q[i] = (uint8_t)((blk[16 + 32 * h + l]", "q[i] = (uint8_t)((blk[16 + 32 * (1 - h) + l]"),
    ("q2k d byte order", "*d = (uint16_t)(blk[80] | (blk[81] << 8));", "*d = (uint16_t)(blk[81] | (blk[80] << 8));"),
    ("q2k d/dmin swapped", "*d = (uint16_t)(blk[80] | (blk[81] << 8));\n    *dmin = (uint16_t)(blk[82] | (blk[83] << 8));",
     "*d = (uint16_t)(blk[82] | (blk[83] << 8));\n    *dmin = (uint16_t)(blk[80] | (blk[81] << 8));"),
    ("q2k nibbles swapped", "d * (double)(sc[s] & 15) * (double)q[i] - dmin * (double)(sc[s] >> 4)",
     "d * (double)(sc[s] >> 4) * (double)q[i] - dmin * (double)(sc[s] & 15)"),
    ("q2k min sign", "d * (double)(sc[s] & 15) * (double)q[i] - dmin", "d * (double)(sc[s] & 15) * (double)q[i] + dmin"),
    ("q2k scale index", "int s = i / 16;", "int s = i / 32;"),
    ("half subnormal exponent", "ldexp((double)m, -24)", "ldexp((double)m, -25)"),
    ("half normal bias", "ldexp((double)(1024 + m), e - 25)", "ldexp((double)(1024 + m), e - 24)"),
    ("half rounding floor", "double m = nearbyint((ldexp(a, -E) - 1.0) * 1024.0);",
     "double m = floor((ldexp(a, -E) - 1.0) * 1024.0);"),
    ("q2k enc step /4", "s[sb] = (mx + m[sb]) / 3.0f;", "s[sb] = (mx + m[sb]) / 4.0f;"),
    ("q2k enc d /16", "uint16_t dh = qso_float_to_half(maxs / 15.0f);", "uint16_t dh = qso_float_to_half(maxs / 16.0f);"),
    ("q2k enc q floor", "qi = (int)clampf_(rintf((x[16 * sb + i] + base) / step), 0.0f, 3.0f);",
     "qi = (int)clampf_(floorf((x[16 * sb + i] + base) / step), 0.0f, 3.0f);"),
    ("q2k enc min unclamped", "m[sb] = mn < 0.0f ? -mn : 0.0f;", "m[sb] = -mn;"),
    ("q4k unpack sc hi", "sc[j] = (uint8_t)((S[j + 4] & 15) | ((S[j - 4] >> 6) << 4));",
     "sc[j] = (uint8_t)((S[j + 4] >> 4) | ((S[j - 4] >> 6) << 4));"),
    ("q4k unpack m hi", "m[j] = (uint8_t)((S[j + 4] >> 4) | ((S[j] >> 6) << 4));",
     "m[j] = (uint8_t)((S[j + 4] & 15) | ((S[j] >> 6) << 4));"),
    ("q4k nibble order", "q[i] = (uint8_t)(l < 32 ? (blk[16 + 32 * c + l] & 15) : (blk[16 + 32 * c + l - 32] >> 4));",
     "q[i] = (uint8_t)(l < 32 ? (blk[16 + 32 * c + l] >> 4) : (blk[16 + 32 * c + l - 32] & 15));"),
    ("q4k d/dmin swapped", "*d = (uint16_t)(blk[0] | (blk[1] << 8));\n    *dmin = (uint16_t)(blk[2] | (blk[3] << 8));",
     "*d = (uint16_t)(blk[2] | (blk[3] << 8));\n    *dmin = (uint16_t)(blk[0] | (blk[1] << 8));"),
    ("q4k sub-block index", "int j = i / 32;\n            w[b * QSO_BLOCK_WEIGHTS + i] = d * (double)sc[j]",
     "int j = i / 64;\n            w[b * QSO_BLOCK_WEIGHTS + i] = d * (double)sc[j]"),
    ("q4k enc sc clamp 31", "int a = df > 0.0f ? (int)clampf_(rintf(s[j] / df), 0.0f, 63.0f) : 0;",
     "int a = df > 0.0f ? (int)clampf_(rintf(s[j] / df), 0.0f, 31.0f) : 0;"),
    ("q4k enc min unclamped", "mm[j] = mn < 0.0f ? -mn : 0.0f;", "mm[j] = -mn;"),
    ("q4k enc d /62", "uint16_t dh = qso_float_to_half(maxs / 63.0f);", "uint16_t dh = qso_float_to_half(maxs / 62.0f);"),
    ("route ties to higher index", "while (j > 0 && l[ord[j - 1]] < l[e])", "while (j > 0 && l[ord[j - 1]] <= l[e])"),
    ("route bias dropped", "if (bias) acc += (double)bias[e];", "if (bias) acc += 0.0;"),
    ("softmax over all E", "for (int j = 0; j < k; j++) den += exp(l[ord[j]] - lmax);",
     "for (int j = 0; j < E; j++) den += exp(l[ord[j]] - lmax);"),
    ("margin from the top", "l[ord[k - 1]] - l[ord[k]]", "l[ord[0]] - l[ord[k]]"),
    ("router transposed", "acc += (double)Wr[(size_t)e * H + h] * xw[h];", "acc += (double)Wr[(size_t)h * E + e] * xw[h];"),
    ("group perm holds tokens", "if (ids[i] == e) perm[pos++] = (int32_t)i;", "if (ids[i] == e) perm[pos++] = (int32_t)(i / k);"),
    ("group offsets not cumulative", "offsets[e + 1] = offsets[e] + counts[e];", "offsets[e + 1] = counts[e];"),
    ("silu sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("routed swiglu operands", "h[r] = silu_(g) * u;", "h[r] = g * silu_(u);"),
    ("shared swiglu operands", "hs[r] = silu_(g) * u;", "hs[r] = g * silu_(u);"),
    ("gate reads up rows", "dequant_row_(fmt, blob + (int64_t)r * rb, H, w);",
     "dequant_row_(fmt, blob + (int64_t)(F + r) * rb, H, w);"),
    ("down reads from the up rows", "const uint8_t *down = blob + 2 * (int64_t)F * rb_h;",
     "const uint8_t *down = blob + (int64_t)F * rb_h;"),
    ("routing weight dropped", "yt[i] += p[(size_t)t * k + j] * ye[i];", "yt[i] += ye[i];"),
    ("shared gate dropped", "y[r] = *gate * acc;", "y[r] = acc;"),
    ("sigmoid sign", "return 1.0 / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(z));"),
    ("shared down transposed", "acc += qso_bf16_to_double(wd[(size_t)r * S + i]) * hs[i];",
     "acc += qso_bf16_to_double(wd[(size_t)i * H + r]) * hs[i];"),
    ("x bf16 read as fp16", "for (int64_t i = 0; i < n; i++) out[i] = qso_bf16_to_double(b[i]);",
     "for (int64_t i = 0; i < n; i++) out[i] = qso_half_to_double(b[i]);"),
    ("steer sign", "yt[i] = yt[i] - scale * (double)d[i] * c;", "yt[i] = yt[i] + scale * (double)d[i] * c;"),
    ("steer dot operand", "for (int i = 0; i < H; i++) c += (double)d[i] * yt[i];",
     "for (int i = 0; i < H; i++) c += (double)d[i] * d[i];"),
    # the Python side of the oracle
    ("threads drop a part", "parts = [todo[i::threads] for i in range(threads)]",
     "parts = [todo[i::threads] for i in range(threads - 1)]", "oracle/__init__.py"),
    ("expert blob gate and up swapped", "np.concatenate([qz(gate).reshape(-1), qz(up).reshape(-1), qz(down).reshape(-1)])",
     "np.concatenate([qz(up).reshape(-1), qz(gate).reshape(-1), qz(down).reshape(-1)])", "oracle/__init__.py"),
    ("steer scale sign in the wrapper", "lib().qso_steer_rows(H, T, _p(dd), float(scale), _p(yy))",
     "lib().qso_steer_rows(H, T, _p(dd), float(-scale), _p(yy))", "oracle/__init__.py"),
]

TESTS = ["tests/test_oracle_q2k.py", "tests/test_oracle_layer.py", "tests/test_oracle_q4k.py",
         "tests/test_oracle_steer.py"]


def mirror():
    if os.path.exists(BASE):
        shutil.rmtree(BASE)
    os.makedirs(BASE)
    shutil.copytree(os.path.join(REPO, "oracle"), os.path.join(BASE, "oracle"),
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    shutil.copytree(os.path.join(REPO, "qs_inputs"), os.path.join(BASE, "qs_inputs"),
                    ignore=shutil.ignore_patterns("__pycache__"))
    shutil.copytree(os.path.join(REPO, "tests"), os.path.join(BASE, "tests"),
                    ignore=shutil.ignore_patterns("__pycache__"))


def main():
    global BASE
    only = sys.argv[1:]
    tmp = tempfile.mkdtemp(prefix="oracle_mutations_")
    BASE = os.path.join(tmp, "m")
    results = []
    for name, old, new, *where in M:
        if only and name not in only:
            continue
        rel = where[0] if where else "oracle/qs_oracle.c"
        src0 = open(os.path.join(REPO, rel)).read()
        n = src0.count(old)
        if n != 1:
            results.append((name, f"BAD PATTERN ({n} matches)"))
            print(name, results[-1][1], flush=True)
            continue
        mirror()
        open(os.path.join(BASE, rel), "w").write(src0.replace(old, new))
        env = dict(os.environ, PYTHONPATH=BASE)
        try:
            r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *TESTS],
                               cwd=BASE, env=env, capture_output=True, text=True, timeout=600)
            caught = r.returncode != 0
            tail = (r.stdout.strip().splitlines() or [""])[-1]
        except subprocess.TimeoutExpired:
            caught, tail = True, "timeout"
        outcome = "caught" if caught else "SURVIVED"
        results.append((name, outcome + " | " + tail))
        print(f"{name}: {outcome} | {tail}", flush=True)
    shutil.rmtree(tmp, ignore_errors=True)
    survivors = [n for n, v in results if not v.startswith("caught")]
    print("\nnot caught:", survivors)
    return 1 if survivors else 0


if __name__ == "__main__":
    sys.exit(main())
