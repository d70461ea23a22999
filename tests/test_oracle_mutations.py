"""The pins can tell a wrong oracle from a right one.

Each case below plants one plausible mistake in a copy of oracle/nf4_oracle.c: a dropped
term, a wrong sign, index or operand, a rounding taken twice, a tie broken the other way, an
off-by-one in a table. The mutated copy is built like the oracle and the whole pin suite
(tests/test_oracle_pins.py) runs against it in a child process. Every mutant must fail at least
one pin. The copies live in a temporary directory; the oracle itself is never modified."""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "nf4_oracle.c")

# (name, text in the oracle, replacement[, which occurrence, counted from 0]): one occurrence
# is replaced, the first unless stated
MUTANTS = [
    ("Phi^-1 without the sqrt(2) of the normal tail",
     "0.5 * erfc(x / sqrt(2.0))", "0.5 * erfc(x / 2.0)"),
    ("NF4 negative half on 9 points instead of 8",
     "-orc_norm_ppf(lin(top, 0.5, 8, j))", "-orc_norm_ppf(lin(top, 0.5, 9, j))"),
    ("int4 absmax codes truncated instead of rounded",
     "float c = nearbyintf(t); /* default rounding mode", "float c = truncf(t); /* default rounding mode"),
    ("nearest-level ties to the higher index",
     "if (d < bd) { bd = d; best = k; }", "if (d <= bd) { bd = d; best = k; }"),
    ("all-zero block coded as level 0 instead of the zero level",
     "codes[b * bs + i] = (uint8_t)zero_idx;", "codes[b * bs + i] = (uint8_t)0;"),
    ("nibble order swapped in packing",
     "packed[j] = (uint8_t)((codes[2 * j] << 4) | (codes[2 * j + 1] & 0xF));",
     "packed[j] = (uint8_t)((codes[2 * j + 1] << 4) | (codes[2 * j] & 0xF));"),
    ("mean of the block scales divided by one block too many",
     "return (float)(total / (double)nb);", "return (float)(total / (double)(nb + 1));"),
    ("scale codes on 128 steps instead of 127",
     "float t = (d / m) * 127.0f;", "float t = (d / m) * 128.0f;"),
    ("rebuilt scale rounded twice (multiply, then add)",
     "return fmaf((float)q, k, mu);", "return (float)q * k + mu;"),
    ("bf16 ties rounded up instead of to even",
     "else pick = ((lo_bits >> 16) & 1u) ? hi_bits : lo_bits;", "else pick = hi_bits;"),
    ("dequantization reads the nibbles in the other order",
     "int c = (i % 2 == 0) ? (byte >> 4) : (byte & 0xF);", "int c = (i % 2 == 0) ? (byte & 0xF) : (byte >> 4);"),
    ("storage size without the fp32 offset",
     "return n / 2 + nb + 4 * ng + 4;", "return n / 2 + nb + 4 * ng;"),
    ("forward without the alpha / r scale on the adapter term",
     "Y_out[ii * N + n] = base + s * lora;", "Y_out[ii * N + n] = base + lora;"),
    ("dX with the adapter term subtracted",
     "dX_out[ii * K + k] = row[k] + s * lora;", "dX_out[ii * K + k] = row[k] - s * lora;"),
    ("dA without the alpha / r scale",
     "dA_out[j * K + k] = s * acc;", "dA_out[j * K + k] = acc;"),
    ("dB from V instead of U",
     "acc += orc_bf16_to_double(G[m * N + n]) * U[m * r + j];",
     "acc += orc_bf16_to_double(G[m * N + n]) * V[m * r + j];"),
    ("merge without the alpha / r scale",
     "orc_bf16_to_double(What[n * K + k]) + s * acc", "orc_bf16_to_double(What[n * K + k]) + acc"),
    ("Philox with nine rounds",
     "for (int round = 0; round < 10; ++round)", "for (int round = 0; round < 9; ++round)"),
    ("dropout without the 1 / (1 - p) rescale of kept elements",
     "double keep_scale = 1.0 / (1.0 - p);", "double keep_scale = 1.0;"),
    ("AdamW without the first moment's bias correction",
     "p[i] -= lr * (m[i] / bc1)", "p[i] -= lr * (m[i])"),
    ("AdamW weight decay not scaled by the learning rate",
     "p[i] *= 1.0 - lr * wd;", "p[i] *= 1.0 - wd;"),
    ("AdamW second moment fed g instead of g^2",
     "(1.0 - b2) * g[i] * g[i];", "(1.0 - b2) * g[i];"),
    ("AdamW epsilon inside the square root",
     "(sqrt(v[i] / bc2) + eps)", "sqrt(v[i] / bc2 + eps)"),
    ("NF4 table divided by the second-largest level",
     "double mx = v[15];", "double mx = v[14];"),
    ("group constant without the mean subtracted",
     "float d = fabsf(s[b] - mu);", "float d = fabsf(s[b]);"),
    ("scale codes truncated instead of rounded",
     "float r = nearbyintf(t);", "float r = truncf(t);"),
    ("fp64 -> bf16 ties rounded up instead of to even",
     "else pick = (fmod(lo / step, 2.0) == 0.0) ? lo : hi;", "else pick = hi;"),
    ("forward reads A transposed",
     "acc += orc_bf16_to_double(X[m * K + k]) * orc_bf16_to_double(A[j * K + k]);",
     "acc += orc_bf16_to_double(X[m * K + k]) * orc_bf16_to_double(A[k * r + j]);"),
    ("dX reads B transposed in V = G B",
     "for (int64_t n = 0; n < N; ++n) acc += orc_bf16_to_double(G[m * N + n]) * orc_bf16_to_double(B[n * r + j]);",
     "for (int64_t n = 0; n < N; ++n) acc += orc_bf16_to_double(G[m * N + n]) * orc_bf16_to_double(B[j * N + n]);"),
    ("dX reads A transposed in V A",
     "for (int64_t j = 0; j < r; ++j) lora += v[j] * orc_bf16_to_double(A[j * K + k]);",
     "for (int64_t j = 0; j < r; ++j) lora += v[j] * orc_bf16_to_double(A[k * r + j]);"),
    ("merge rounded through fp32 (twice)",
     "out[n * K + k] = orc_bf16_round_d(orc_bf16_to_double(What[n * K + k]) + s * acc);",
     "out[n * K + k] = orc_bf16_round((float)(orc_bf16_to_double(What[n * K + k]) + s * acc));"),
    ("Philox with the first Weyl constant for both key words",
     "k1 += 0xBB67AE85u;", "k1 += 0x9E3779B9u;"),
    ("dropout takes word 0 of every block",
     "D[e] = (w[e % 4] >= thr) ? keep_scale : 0.0;", "D[e] = (w[0] >= thr) ? keep_scale : 0.0;"),
    ("dropout dX without the mask on the adapter term",
     "dX_out[ii * K + k] = row[k] + D[m * K + k] * s * lora;", "dX_out[ii * K + k] = row[k] + s * lora;"),
    ("dropout dA without the mask on X",
     "acc += V[m * r + j] * orc_bf16_to_double(X[m * K + k]) * D[m * K + k];",
     "acc += V[m * r + j] * orc_bf16_to_double(X[m * K + k]);"),
    ("int4 absmax from the signed maximum",
     "for (int64_t i = 0; i < n; ++i) if (fabsf(w[i]) > am) am = fabsf(w[i]);",
     "for (int64_t i = 0; i < n; ++i) if (w[i] > am) am = w[i];"),
    ("NF4 block absmax from the signed maximum",
     "for (int64_t i = 0; i < bs; ++i) if (fabsf(blk[i]) > am) am = fabsf(blk[i]);",
     "for (int64_t i = 0; i < bs; ++i) if (blk[i] > am) am = blk[i];"),
    ("nearest level by signed difference",
     "        float d = fabsf(x - levels[k]);", "        float d = x - levels[k];"),
    ("degenerate group coded 1 instead of 0",
     "if (m == 0.0f) { q[b] = 0; continue; }", "if (m == 0.0f) { q[b] = 1; continue; }"),
    ("group sums of the mean accumulated in fp32",
     "        double acc = 0.0;\n        int64_t b1", "        float acc = 0.0f;\n        int64_t b1"),
    ("dequantization always takes group 0's constant",
     "int64_t b = i / 64, g = b / 256;", "int64_t b = i / 64, g = 0 * b;"),
    ("rebuilt scale step c2 / 128",
     "float k = c2 / 127.0f;", "float k = c2 / 128.0f;"),
    ("fp32 -> bf16 never rounds up past a non-tie",
     "else if (dhi < dlo) pick = hi_bits;", "else if (dhi < 0.0) pick = hi_bits;"),
    ("forward scale alpha / (r + 1)",
     "double s = alpha / (double)r;", "double s = alpha / (double)(r + 1);"),
    ("dA from U instead of V",
     "acc += V[m * r + j] * orc_bf16_to_double(X[m * K + k]);",
     "acc += U[m * r + j] * orc_bf16_to_double(X[m * K + k]);"),
    ("Philox mixes the key words the other way round",
     "uint32_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;",
     "uint32_t n0 = hi1 ^ c1 ^ k1, n1 = lo1, n2 = hi0 ^ c3 ^ k0, n3 = lo0;"),
    ("dropout threshold on 2^31",
     "uint32_t thr = (uint32_t)floor(p * 4294967296.0);", "uint32_t thr = (uint32_t)floor(p * 2147483648.0);"),
    ("dropout counter with the element index and the offset swapped",
     "uint32_t ctr[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), (uint32_t)offset, (uint32_t)(offset >> 32)};",
     "uint32_t ctr[4] = {(uint32_t)offset, (uint32_t)(offset >> 32), (uint32_t)blk, (uint32_t)(blk >> 32)};"),
    ("AdamW without the second moment's bias correction",
     "(sqrt(v[i] / bc2) + eps)", "(sqrt(v[i]) + eps)"),
    ("AdamW first moment without the (1 - beta1) factor",
     "m[i] = b1 * m[i] + (1.0 - b1) * g[i];", "m[i] = b1 * m[i] + g[i];"),
    ("merge reads A transposed",
     "acc += orc_bf16_to_double(B[n * r + j]) * orc_bf16_to_double(A[j * K + k]);",
     "acc += orc_bf16_to_double(B[n * r + j]) * orc_bf16_to_double(A[k * r + j]);"),
    ("merge reads B transposed",
     "acc += orc_bf16_to_double(B[n * r + j]) * orc_bf16_to_double(A[j * K + k]);",
     "acc += orc_bf16_to_double(B[j * N + n]) * orc_bf16_to_double(A[j * K + k]);"),
    ("sampled dB columns without the alpha / r scale",
     "dB_cols[jj * N + n] = s * acc;", "dB_cols[jj * N + n] = acc;"),
    ("dropout dB from the unmasked U",
     "au += orc_bf16_to_double(X[m * K + k]) * D[m * K + k] * orc_bf16_to_double(A[j * K + k]);",
     "au += orc_bf16_to_double(X[m * K + k]) * orc_bf16_to_double(A[j * K + k]);"),
    ("int4 reconstruction on 8 steps",
     "w_hat[i] = (c / 7.0f) * am;", "w_hat[i] = (c / 8.0f) * am;"),
    ("MSE of the sum instead of the residual",
     "double e = (double)(r - w[i]);", "double e = (double)(r + w[i]);"),
    ("fp64 -> bf16 subnormal spacing one binade too fine",
     "if (q < -133) q = -133;", "if (q < -134) q = -134;"),
    ("fp64 -> bf16 overflows one binade early",
     "if (pick >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);",
     "if (pick >= ldexp(1.0, 127)) return (uint16_t)(sign | 0x7F80);"),
    ("fp32 -> bf16 overflow distance taken to the infinity pattern",
     "double dhi = isinf(hi) ? fabs(ldexp(1.0, 128) - fabs((double)x)) : fabs((double)hi - (double)x);",
     "double dhi = fabs((double)hi - (double)x);"),
    ("mean's tree pairs elements i and i + len / 2",
     "t[i] = t[2 * i] + t[2 * i + 1];", "t[i] = t[i] + t[i + len / 2];"),
    ("NF4 top probability 0.96",
     "const double top = 0.9677083;", "const double top = 0.96;"),
    ("Phi^-1 without the sign for p < 1/2",
     "double sign = (p < 0.5) ? -1.0 : 1.0;", "double sign = 1.0;"),
    ("linspace divided by n instead of n - 1",
     "return a + (b - a) * (double)i / (double)(n - 1); }", "return a + (b - a) * (double)i / (double)n; }"),
    ("NF4 table sorted descending",
     "while (j >= 0 && v[j] > x)", "while (j >= 0 && v[j] < x)"),
    ("unpacking takes the low nibble for the first code",
     "codes[2 * j] = (uint8_t)(packed[j] >> 4);", "codes[2 * j] = (uint8_t)(packed[j] & 0xF);"),
    ("AdamW bias correction one step behind",
     "double bc1 = 1.0 - pow(b1, (double)t)", "double bc1 = 1.0 - pow(b1, (double)(t + 1))"),
    ("dropout key without the seed's high half",
     "uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};", "uint32_t key[2] = {(uint32_t)seed, 0u};"),
    ("dX reads W^ transposed",
     "for (int64_t k = 0; k < K; ++k) row[k] += g * orc_bf16_to_double(What[n * K + k]);",
     "for (int64_t k = 0; k < K; ++k) row[k] += g * orc_bf16_to_double(What[k * N + n]);"),
    ("forward reads W^ transposed",
     "for (int64_t k = 0; k < K; ++k) base += orc_bf16_to_double(X[m * K + k]) * orc_bf16_to_double(What[n * K + k]);",
     "for (int64_t k = 0; k < K; ++k) base += orc_bf16_to_double(X[m * K + k]) * orc_bf16_to_double(What[k * N + n]);"),
    ("dropout forward applies the mask to the base term too",
     "for (int64_t k = 0; k < K; ++k) base += orc_bf16_to_double(X[m * K + k]) * orc_bf16_to_double(What[n * K + k]);",
     "for (int64_t k = 0; k < K; ++k) base += orc_bf16_to_double(X[m * K + k]) * D[m * K + k] * "
     "orc_bf16_to_double(What[n * K + k]);", 1),
    ("dropout forward reads B transposed",
     "for (int64_t j = 0; j < r; ++j) lora += u[j] * orc_bf16_to_double(B[n * r + j]);",
     "for (int64_t j = 0; j < r; ++j) lora += u[j] * orc_bf16_to_double(B[j * N + n]);", 1),
    ("sampled dA rows without the alpha / r scale",
     "dA_rows[jj * K + k] = s * acc;", "dA_rows[jj * K + k] = acc;"),
    ("sampled grads read B transposed in V",
     "for (int64_t n = 0; n < N; ++n) av += orc_bf16_to_double(G[m * N + n]) * orc_bf16_to_double(B[n * r + j]);",
     "for (int64_t n = 0; n < N; ++n) av += orc_bf16_to_double(G[m * N + n]) * orc_bf16_to_double(B[j * N + n]);", 1),
    ("dropout grads read B transposed in V",
     "for (int64_t n = 0; n < N; ++n) av += orc_bf16_to_double(G[m * N + n]) * orc_bf16_to_double(B[n * r + j]);",
     "for (int64_t n = 0; n < N; ++n) av += orc_bf16_to_double(G[m * N + n]) * orc_bf16_to_double(B[j * N + n]);", 2),
    ("dropout dB without the alpha / r scale",
     "dB_out[n * r + j] = s * acc;", "dB_out[n * r + j] = acc;", 1),
    ("dropout dA without the alpha / r scale",
     "dA_out[j * K + k] = s * acc;", "dA_out[j * K + k] = acc;", 1),
    ("unpacking swaps the nibbles of the second code",
     "codes[2 * j + 1] = (uint8_t)(packed[j] & 0xF);", "codes[2 * j + 1] = (uint8_t)(packed[j] >> 4);"),
]


def _mutate(src, old, new, nth=0):
    at = -1
    for _ in range(nth + 1):
        at = src.find(old, at + 1)
        assert at >= 0, f"mutation site not found: {old!r} (occurrence {nth})"
    return src[:at] + new + src[at + len(old):]


def _run_mutant(tmp, i, mutant, src):
    path = os.path.join(tmp, f"mutant{i}.c")
    so = os.path.join(tmp, f"libmutant{i}.so")
    with open(path, "w") as f:
        f.write(_mutate(src, *mutant[1:]))
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-o", so,
                    path, "-lm"], check=True, capture_output=True)
    env = dict(os.environ, ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-x", "-q",
                        "-p", "no:cacheprovider"], env=env, cwd=ROOT, capture_output=True, text=True, timeout=900)
    return r.returncode


def test_every_planted_mistake_fails_a_pin(tmp_path):
    if os.environ.get("ORACLE_LIB"):
        pytest.skip("this process already runs another build of the oracle")
    src = open(SRC).read()
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        codes = list(ex.map(lambda a: _run_mutant(str(tmp_path), a[0], a[1], src), enumerate(MUTANTS)))
    survivors = [m[0] for m, rc in zip(MUTANTS, codes) if rc == 0]
    assert not survivors, f"mutants no pin catches: {survivors}"
    # a failing pin (exit 1), not a crash or a usage error, is what stopped each run
    assert all(rc == 1 for rc in codes), list(zip([m[0] for m in MUTANTS], codes))
