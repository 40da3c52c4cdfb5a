"""Mutation check of the oracle's pins: plant one plausible mistake at a time
in a copy of the oracle's C source (a flipped sign, a wrong tie rule, a
transposed index, a wrong constant, a wrong layout size ...), build it, and
run the pin suite against it in a child process.  Every mutant must fail at
least one pin; a mutant that passes would mean the pins cannot tell that
mistake from the method.  Mistakes are planted on the CPU, in the oracle
only."""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kv_oracle.c")

# (name, text in the oracle, replacement)
MUTANTS = [
    ("fwht sign", "x[j + h] = a - b;", "x[j + h] = b - a;"),
    ("fwht pairing", "double a = x[j], b = x[j + h];", "double a = x[j], b = x[(j + h) % d];\n                (void)0; a = x[j]; b = x[j ^ h ^ (h > 1 ? 1 : 0)];"),
    ("threshold tie to lower cell", "if (t[j] <= u) code++;", "if (t[j] < u) code++;"),
    ("centroid typo", "-0.7560, -0.2451, 0.2451, 0.7560,", "-0.7560, -0.2451, 0.2451, 0.7650,"),
    ("sigma normaliser", "double sigma = nrm / sqrt((double)d);", "double sigma = nrm / (double)d;"),
    ("u normalised by sigma", "? y[i] / nrm : 0.0;", "? y[i] / (nrm / sqrt((double)d)) : 0.0;"),
    ("k scale 128", "return (float)(m / 127.0);", "return (float)(m / 128.0);"),
    ("k rounding ties away", "double q = nearbyint(k / (double)s);", "double q = round(k / (double)s);"),
    # (A -128 lower clamp would be an equivalent mutant: with s = fl(m/127),
    # |k/s| <= 127.00001, so no input reaches it.)
    ("k decode divides", "return orc_f64_to_bf16((double)q * (double)s);", "return orc_f64_to_bf16((double)q / (double)s);"),
    ("pack3 bit order", "w |= (uint32_t)(codes[8 * g + j] & 7u) << (3 * j);", "w |= (uint32_t)(codes[8 * g + j] & 7u) << (3 * (7 - j));"),
    ("decode rescale", "out[i] = orc_f64_to_bf16(sig * z[i] / rs);", "out[i] = orc_f64_to_bf16(sig * z[i] / (double)d);"),
    ("bf16 ties away", "double r = nearbyint(scaled);", "double r = floor(scaled + 0.5);"),
    ("fp16 subnormal scale", "return sign | (uint16_t)ldexp(r, 24);", "return sign | (uint16_t)ldexp(r, 23);"),
    ("lloyd mean sign", "double m = (pa - pb) / (Phi(b) - Phi(a));", "double m = (pb - pa) / (Phi(b) - Phi(a));"),
    ("group scale levels", "double qmax = (double)((1 << b) - 1);", "double qmax = (double)(1 << b);"),
    ("group zero point max", "uint16_t zb = orc_f64_to_f16(mn);", "uint16_t zb = orc_f64_to_f16(mx);"),
    ("group bit order", "int bit = j * b + k;\n                out[bit >> 3]", "int bit = j * b + (b - 1 - k);\n                out[bit >> 3]"),
    ("card params per group", "+ (uint64_t)H * (uint64_t)(d / 32) * 4ull);", "+ (uint64_t)H * (uint64_t)(d / 32) * 2ull);"),
    ("pool sigma offset", "g.sec_sigma = al256(g.sec_v + nv * (uint64_t)(3 * d / 8));", "g.sec_sigma = al256(g.sec_v + nv * (uint64_t)(d / 2));"),
    ("k absmax skips sign", "double a = fabs(orc_bf16_to_f64(k[i]));", "double a = orc_bf16_to_f64(k[i]);"),
    ("attend GQA head map", "const int j = aj % n_q_heads;\n        const int h = j / grp;",
     "const int j = aj % n_q_heads;\n        const int h = j % H;"),
    ("attend lse drops max", "lse[aj] = mx + log(sum);\n        free(sc);\n    }",
     "lse[aj] = log(sum);\n        free(sc);\n    }"),
    ("realign shift reversed", "const double delta = (double)(pos_dst - pos_src);",
     "const double delta = (double)(pos_src - pos_dst);"),
    ("realign sine sign", "row[i] = orc_f64_to_bf16(a * cs[i] - c * sn[i]);",
     "row[i] = orc_f64_to_bf16(a * cs[i] + c * sn[i]);"),
    ("realign adjacent pairs", "double a = x[i], c = x[i + half];", "double a = x[i], c = x[i ^ 1];"),
    ("realign frequency order", "double phi = delta * (double)w[i];", "double phi = delta * (double)w[half - 1 - i];"),
    ("realign drops zero point", "x[32 * gi + i] = (double)q[i] * sc + z;", "x[32 * gi + i] = (double)q[i] * sc;"),
    ("q8 scale divisor 128", "uint16_t sb = orc_f64_to_f16(m / 127.0);", "uint16_t sb = orc_f64_to_f16(m / 128.0);"),
    ("q8 ties away from zero", "double q = nearbyint(k / s);", "double q = round(k / s);"),
    ("q8 scales per layer offset", "uint8_t *ks = pool + g.off_kscales + (uint64_t)l * nb * 2u;",
     "uint8_t *ks = pool + g.off_kscales + (uint64_t)l * nb;"),
    ("q8 attend uses tensor scale", "sk = orc_f16_to_f64(sb);", "sk = (double)s;"),
    ("lora head slice by query head", "orc_bf16_to_f64(ba[(uint64_t)k * H * d + (uint64_t)h * d + i]);",
     "orc_bf16_to_f64(ba[(uint64_t)k * H * d + (uint64_t)(j % H) * d + i]);"),
    ("lora up-projection transposed", "orc_bf16_to_f64(ba[(uint64_t)k * H * d + (uint64_t)h * d + i]);",
     "orc_bf16_to_f64(ba[((uint64_t)h * d + i) * (uint64_t)rank + k]);"),
    ("lora first agent's B for all", "const uint16_t *ba = lora_b + (uint64_t)a * (uint64_t)rank * (uint64_t)H * d;",
     "const uint16_t *ba = lora_b;"),
    ("lora low-rank cache transposed", "v += orc_bf16_to_f64(vlr[(uint64_t)t * rank + k]) *",
     "v += orc_bf16_to_f64(vlr[(uint64_t)k * T + t]) *"),
    ("q8 decode reads next block", "kk[i] = orc_k_block_decode(q, sb);",
     "memcpy(&sb, ks + 2u * ((uint64_t)n * (uint64_t)(d / 32) + (uint64_t)((i / 32 + 1) % (d / 32))), 2);\n                    kk[i] = orc_k_block_decode(q, sb);"),
]


def _build(text, out):
    src = out + ".c"
    with open(src, "w") as f:
        f.write(text)
    r = subprocess.run(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off", "-fopenmp", src,
                        "-o", out, "-lm"], capture_output=True, text=True)
    if r.returncode != 0:  # no OpenMP on this host
        r = subprocess.run(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off", src, "-o", out,
                            "-lm"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def _run_mutant(old, new):
    """Build the oracle with one mistake planted and run the pin suite against
    it in a child process; returns (site count, return code, output tail)."""
    text = open(SRC).read()
    count = text.count(old)
    if count != 1:
        return count, None, ""
    with tempfile.TemporaryDirectory() as tmp:
        lib = os.path.join(tmp, "mutant.so")
        _build(text.replace(old, new), lib)
        env = dict(os.environ, KV_ORACLE_LIB=lib, PYTHONPATH=ROOT, OMP_NUM_THREADS="2")
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                            os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                           capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)
    return count, r.returncode, r.stdout[-2000:]


@pytest.fixture(scope="module")
def mutant_results():
    """Every mutant's run, eight child processes at a time."""
    import concurrent.futures as cf
    with cf.ThreadPoolExecutor(max_workers=8) as ex:
        futs = {name: ex.submit(_run_mutant, old, new) for name, old, new in MUTANTS}
        return {name: f.result() for name, f in futs.items()}


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, mutant_results):
    count, rc, out = mutant_results[name]
    assert count == 1, "mutation site found %d times, not once" % count
    assert rc != 0, "mutant '%s' passed every pin:\n%s" % (name, out)
