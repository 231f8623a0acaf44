"""The oracle's pins must fail on plausible mistakes.

Each mutant below is the oracle source with one plausible slip planted (on the CPU, in a
temporary copy). The mutant is compiled and the pin suite is run against it in a
subprocess; the suite must fail. A mutant that survives means some part of the oracle is
not pinned by anything but itself.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "zero_oracle.c")

# (name, original text, planted text)
MUTANTS = [
    ("rank order reversed", "for (int32_t r = 0; r < M; ++r) acc = acc + orc_bf16_to_f32(g[r][o]);",
     "for (int32_t r = M - 1; r >= 0; --r) acc = acc + orc_bf16_to_f32(g[r][o]);"),
    ("sum instead of average", "    return acc * inv_M;", "    return acc;"),
    ("accumulator starts at -0", "float acc = 0.0f; /* +0", "float acc = -0.0f; /* +0"),
    ("shard index transposed", "int64_t in_bucket = (int64_t)r * b_S[b] + j;\n                int64_t o = b_off[b] + in_bucket;",
     "int64_t in_bucket = j * (int64_t)M + r;\n                int64_t o = b_off[b] + in_bucket;"),
    ("padding counted in the streamed norm", "if (o - b_off[b] < b_n[b]) {", "if (o >= 0) {"),
    ("no bias correction of m", "k.step_size = (float)(h->lr / bc1);", "k.step_size = (float)(h->lr);"),
    ("no bias correction of v", "k.inv_sqrt_bc2 = (float)(1.0 / sqrt(bc2));", "k.inv_sqrt_bc2 = 1.0f;"),
    ("weight decay sign", "k.decay = (float)(1.0 - h->lr * h->weight_decay);",
     "k.decay = (float)(1.0 + h->lr * h->weight_decay);"),
    ("eps inside the square root", "float den = sqrtf(v1) * k->inv_sqrt_bc2 + k->eps;",
     "float den = sqrtf(v1 + k->eps) * k->inv_sqrt_bc2;"),
    ("betas swapped", "float m1 = k->b1 * (*m) + k->c1 * g;", "float m1 = k->b2 * (*m) + k->c2 * g;"),
    ("clip scale not applied", "    float g = s * ghat;", "    float g = ghat;"),
    ("clip when below threshold", "if (norm > max_grad_norm) return (float)(max_grad_norm / norm);",
     "if (norm < max_grad_norm) return (float)(max_grad_norm / norm);"),
    ("round toward zero", "u += 0x7FFFu + keep_odd;", "u += 0u * keep_odd;"),
    ("ties away from zero", "u += 0x7FFFu + keep_odd;", "u += 0x8000u + 0u * keep_odd;"),
    ("padding not rounded up", "b_S[b] = ((b_n[b] + unit - 1) / unit) * A;", "b_S[b] = (b_n[b] / unit) * A;"),
    ("bucket cap ignored", "cur_bytes + bytes > bucket_bytes);", "cur_bytes + bytes > 2 * bucket_bytes);"),
    ("gather to padded place", "if (in_bucket < b_n[b]) dst[ubase + in_bucket] = shard_bf16[r][base + j];",
     "if (in_bucket < b_n[b]) dst[base * 0 + in_bucket + b * 1] = shard_bf16[r][base + j];"),
    ("groups summed flat", "        for (int32_t k = 0; k < K; ++k) part = part + orc_bf16_to_f32(g[grp * K + k][o]);\n        acc = acc + part;",
     "        for (int32_t k = 0; k < K; ++k) acc = acc + orc_bf16_to_f32(g[grp * K + k][o]);\n        part = part + acc;"),
    ("saved v dropped on resume", "var[r][base + j] = (real && v_init) ? v_init[u] : 0.0f;",
     "var[r][base + j] = 0.0f;"),
    ("saved m and v swapped on resume", "mom[r][base + j] = (real && m_init) ? m_init[u] : 0.0f;",
     "mom[r][base + j] = (real && v_init) ? v_init[u] : 0.0f;"),
    ("nonfinite not skipped", "if (!isfinite(norm)) skipped = 1;\n        else s = orc_clip_scale(norm, h->max_grad_norm);\n    }\n    *scale_out = s;",
     "s = orc_clip_scale(norm, h->max_grad_norm);\n    }\n    *scale_out = s;"),
]


def _run_mutant(name, old, new, tmpdir):
    src = open(SRC).read()
    if src.count(old) < 1:
        return f"mutation site for '{name}' not found"
    d = os.path.join(tmpdir, "".join(c if c.isalnum() else "_" for c in name))
    os.makedirs(d)
    cfile = os.path.join(d, "mutant.c")
    with open(cfile, "w") as f:
        f.write(src.replace(old, new, 1))
    lib = os.path.join(d, "libmutant.so")
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                    "-o", lib, cfile, "-lm"], check=True)
    env = dict(os.environ, ZERO_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-k", "not exhaustive"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return None if r.returncode != 0 else f"mutant '{name}' survived the pins"


def test_pins_kill_every_mutant(tmp_path):
    workers = max(1, min(len(MUTANTS), os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        results = list(ex.map(lambda m: _run_mutant(*m, str(tmp_path)), MUTANTS))
    problems = [r for r in results if r]
    assert not problems, "\n".join(problems)
