"""The oracle pins have teeth: plant a plausible mistake in a copy of the
oracle's C source (on the CPU), rebuild it, and check that the pin suite now
fails.  Each mutant is one slip a reader of the pages could make."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "q4_oracle.c")

MUTANTS = [
    ("q4_0 nibble order interleaved",
     "int q = (j < 16) ? (qs[j] & 0x0f) : (qs[j - 16] >> 4);",
     "int q = (qs[j / 2] >> (4 * (j & 1))) & 0x0f;"),
    ("q4_0 offset dropped", "w[b * 32 + j] = d * (double)(q - 8);", "w[b * 32 + j] = d * (double)q;"),
    ("q4_0 offset sign", "w[b * 32 + j] = d * (double)(q - 8);", "w[b * 32 + j] = d * (double)(8 - q);"),
    ("fp16 scale byte order", "double d = q4o_half((uint16_t)(blk[0] | (blk[1] << 8)));\n        const uint8_t *qs",
     "double d = q4o_half((uint16_t)(blk[1] | (blk[0] << 8)));\n        const uint8_t *qs"),
    ("fp16 exponent bias", "v = ldexp((double)(f | 0x400), e - 25);", "v = ldexp((double)(f | 0x400), e - 24);"),
    ("fp16 subnormal scale", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    ("bf16 exponent bias", "v = ldexp((double)(f | 0x80), e - 134);", "v = ldexp((double)(f | 0x80), e - 133);"),
    ("affine nibble order", "int q = (e & 1) ? (byte >> 4) : (byte & 0x0f);",
     "int q = (e & 1) ? (byte & 0x0f) : (byte >> 4);"),
    ("affine min sign", "w[e] = sg * (double)q + mg;", "w[e] = sg * (double)q - mg;"),
    ("affine min dropped", "w[e] = sg * (double)q + mg;", "w[e] = sg * (double)q;"),
    ("activation row ignored", "acc += wrow[e] * xr[e];", "acc += wrow[e] * x[e];"),
    ("rmsnorm sum not mean", "double rms = sqrt(ss / (double)k + eps);", "double rms = sqrt(ss + eps);"),
    ("rmsnorm eps outside sqrt", "double rms = sqrt(ss / (double)k + eps);",
     "double rms = sqrt(ss / (double)k) + eps;"),
    ("rmsnorm gamma dropped", "xhat[r * k + e] = xr[e] / rms * gamma[e];", "xhat[r * k + e] = xr[e] / rms;"),
    ("silu sign", "return t / (1.0 + exp(-t));", "return t / (1.0 + exp(t));"),
    ("swiglu factors swapped", "h[i] = q4o_silu(g[i]) * u[i];", "h[i] = q4o_silu(u[i]) * g[i];"),
    ("residual subtracted", "out[i] = a[i] + b[i];", "out[i] = a[i] - b[i];"),
    ("argmax tie to last", "if (v[i] > v[best])", "if (v[i] >= v[best])"),
    ("q8_0 bytes read unsigned", "int q = blk[2 + j] < 128 ? blk[2 + j] : blk[2 + j] - 256;",
     "int q = blk[2 + j];"),
    ("q8_0 block stride", "const uint8_t *blk = r + b * 34;", "const uint8_t *blk = r + b * 32;"),
    ("q8_0 scale byte order", "double d = q4o_half((uint16_t)(blk[0] | (blk[1] << 8)));\n        for (int j = 0; j < 32; ++j) {\n            int q = blk[2 + j]",
     "double d = q4o_half((uint16_t)(blk[1] | (blk[0] << 8)));\n        for (int j = 0; j < 32; ++j) {\n            int q = blk[2 + j]"),
    ("q4_k min sign", "w[b * 256 + e] = d * (double)sc * (double)q - dmin * (double)mn;",
     "w[b * 256 + e] = d * (double)sc * (double)q + dmin * (double)mn;"),
    ("q4_k d and dmin swapped", "double d = q4o_half((uint16_t)(blk[0] | (blk[1] << 8)));\n        double dmin",
     "double d = q4o_half((uint16_t)(blk[2] | (blk[3] << 8)));\n        double dmin"),
    ("q4_k nibble halves swapped", "int q = (j & 1) ? (byte >> 4) : (byte & 0x0f);",
     "int q = (j & 1) ? (byte & 0x0f) : (byte >> 4);"),
    ("q4_k nibbles interleaved", "int byte = qs[32 * (j / 2) + l];", "int byte = qs[e / 2];"),
    ("q4_k high scale bits from the min byte", "*sc = (sb[j + 4] & 0x0f) | ((sb[j - 4] >> 6) << 4);",
     "*sc = (sb[j + 4] & 0x0f) | ((sb[j] >> 6) << 4);"),
    ("q4_k high min nibble", "*mn = (sb[j + 4] >> 4) | ((sb[j] >> 6) << 4);",
     "*mn = (sb[j + 4] & 0x0f) | ((sb[j] >> 6) << 4);"),
    ("q4_k low mins from the scale bytes", "*mn = sb[j + 4] & 63;", "*mn = sb[j] & 63;"),
    ("q1 sign convention", "w[b * 128 + e] = bit ? d : -d;", "w[b * 128 + e] = bit ? -d : d;"),
    ("q1 bits most significant first", "int bit = (blk[2 + e / 8] >> (e % 8)) & 1;",
     "int bit = (blk[2 + e / 8] >> (7 - e % 8)) & 1;"),
    ("q1 bits start at the scale", "int bit = (blk[2 + e / 8] >> (e % 8)) & 1;",
     "int bit = (blk[e / 8] >> (e % 8)) & 1;"),
    ("q1 superblock stride", "const uint8_t *blk = r + b * 18;\n        double d = q4o_half((uint16_t)(blk[0] | (blk[1] << 8)));\n        for (int e = 0; e < 128",
     "const uint8_t *blk = r + b * 16;\n        double d = q4o_half((uint16_t)(blk[0] | (blk[1] << 8)));\n        for (int e = 0; e < 128"),
    ("attn kv head by modulo", "int64_t hk = h / G;", "int64_t hk = h % Hkv;"),
    ("attn window one short", "int64_t lo = (window > 0 && total > window) ? total - window : 0;",
     "int64_t lo = (window > 0 && total > window) ? total - window + 1 : 0;"),
    ("attn scale dropped", "p[t] = scale * s;", "p[t] = s;"),
    ("attn softmax unnormalised", "acc += p[t] / z * v;", "acc += p[t] * v;"),
    ("attn appended k not rotated", "if (cosv)\n            q4o_rope_apply(kh,", "if (0)\n            q4o_rope_apply(kh,"),
    ("rope sign", "x[j] = a * c[j] - b * s[j];", "x[j] = a * c[j] + b * s[j];"),
    ("rope angle exponent", "pow(rope_theta, 2.0 * (double)j / (double)d)", "pow(rope_theta, (double)j / (double)d)"),
    ("halfset streams swapped", "x[r * k + 2 * i] = q4o_half(xe[r * (k / 2) + i]);",
     "x[r * k + 2 * i] = q4o_half(xo[r * (k / 2) + i]);"),
    ("halfset rows concatenated", "x[r * k + 2 * i + 1] = q4o_half(xo[r * (k / 2) + i]);",
     "x[r * k + k / 2 + i] = q4o_half(xo[r * (k / 2) + i]);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, name
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-shared", "-fPIC",
                           "-o", str(so), str(mut), "-lm"])
    env = dict(os.environ, Q4_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "pins did not catch mutant: " + name
