"""Planted mistakes in the oracle, on the CPU: each copy of oracle.c with one
plausible mistake (a rounding rule, a bias, a threshold, an index, an
operand, an order) is compiled on its own and must fail at least one pin in
test_oracle_pins.py; an unmodified copy built the same way must pass them
all. The mutants run in subprocesses with ORACLE_LIBRARY pointing at their
library, so the committed oracle is never touched."""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (name, text in oracle.c, replacement, which occurrence). Left out because no
# input can tell it apart: removing the e4m3 encoder's final clamp of codes
# above 0x7E (below 448 the grid step is 32, so nothing there rounds past 448).
MUTATIONS = [
    ("bf16 ties round up", "(lo == 0x8000u && (hi & 1u))", "(lo == 0x8000u)", 0),
    ("e4m3 ties round up", "double m = rint(ldexp(a, 3 - E));", "double m = floor(ldexp(a, 3 - E) + 0.5);", 0),
    ("e4m3 subnormal threshold", "if (a < ldexp(1.0, -6)) {", "if (a < ldexp(1.0, -7)) {", 0),
    ("e5m2 ties round up", "double m = rint(ldexp(a, 2 - E));", "double m = floor(ldexp(a, 2 - E) + 0.5);", 0),
    ("e5m2 encoder bias", "int code = ((E + 15) << 2) | ((int)m - 4);", "int code = ((E + 14) << 2) | ((int)m - 4);", 0),
    ("e5m2 decoder bias", "v = ldexp(1.0 + m / 4.0, field - 15);", "v = ldexp(1.0 + m / 4.0, field - 14);", 0),
    ("e5m2 subnormal threshold", "if (a < ldexp(1.0, -14)) {", "if (a < ldexp(1.0, -15)) {", 0),
    ("rank of an expert by e mod R", "mask[e / L] = 1;", "mask[e % R] = 1;", 0),
    ("rank counts slots, not tokens", "mask[e / L] = 1;", "mask[e / L] += 1;", 0),
    ("inclusive expert offsets",
     "        expert_offsets[e] = (int32_t)run;\n        num_tokens_per_expert[e] = (int32_t)cnt64[e];",
     "        expert_offsets[e] = (int32_t)(run + cnt64[e]);\n        num_tokens_per_expert[e] = (int32_t)cnt64[e];", 0),
    ("rows in descending k",
     "for (int k = 0; k < K; ++k) {\n            int64_t e = topk_idx[t * K + k];\n"
     "            if (e < 0 || e >= E) { row_of_slot[t * K + k] = -1; continue; }",
     "for (int k = K - 1; k >= 0; --k) {\n            int64_t e = topk_idx[t * K + k];\n"
     "            if (e < 0 || e >= E) { row_of_slot[t * K + k] = -1; continue; }", 0),
    ("combine multiply and add rounded apart", "acc = fmaf(wk, orc_bf16_to_f32(y[(int64_t)row * H + h]), acc);",
     "acc = wk * orc_bf16_to_f32(y[(int64_t)row * H + h]) + acc;", 0),
    ("quantise by the reciprocal", "float v = orc_bf16_to_f32(xrow[b * 128 + i]) / scale;",
     "float v = orc_bf16_to_f32(xrow[b * 128 + i]) * (1.0f / scale);", 0),
    ("e5m2 quantise by the reciprocal",
     "qrow[b * 128 + i] = orc_f32_to_e5m2(orc_bf16_to_f32(xrow[b * 128 + i]) / scale);",
     "qrow[b * 128 + i] = orc_f32_to_e5m2(orc_bf16_to_f32(xrow[b * 128 + i]) * (1.0f / scale));", 0),
    ("e4m3 largest finite 480", "float scale = amax / 448.0f;", "float scale = amax / 480.0f;", 0),
    ("e5m2 largest finite 49152", "float scale = amax / 57344.0f;", "float scale = amax / 49152.0f;", 0),
    ("power-of-two scale not rounded up", "float scale = orc_pow2_ceil(amax / 448.0f);",
     "float scale = amax / 448.0f;", 0),
    ("e4m3 UE8M0 byte off by one", "sbytes[b] = (uint8_t)(ex - 1 + 127);", "sbytes[b] = (uint8_t)(ex + 127);", 0),
    ("e5m2 UE8M0 byte off by one", "sbytes[b] = (uint8_t)(ex - 1 + 127);", "sbytes[b] = (uint8_t)(ex + 127);", 1),
    ("e4m3 UE8M0 without the 2^-127 floor", "if (scale < ldexpf(1.0f, -127)) scale = ldexpf(1.0f, -127);", "", 0),
    ("e5m2 UE8M0 without the 2^-127 floor", "if (scale < ldexpf(1.0f, -127)) scale = ldexpf(1.0f, -127);", "", 1),
    ("combine backward drops the weight", "orc_f32_to_bf16(wk * g)", "orc_f32_to_bf16(g)", 0),
    ("weight gradient against a reversed row",
     "dot += (double)g * (double)orc_bf16_to_f32(y[(int64_t)row * H + h]);",
     "dot += (double)g * (double)orc_bf16_to_f32(y[(int64_t)row * H + (H - 1 - h)]);", 0),
    ("dispatch backward gathers the wrong weight",
     "grad_topk_weights[s] = row >= 0 ? grad_recv_weights[row] : 0.0f;",
     "grad_topk_weights[s] = row >= 0 ? grad_recv_weights[s % (row + 1)] : 0.0f;", 0),
    ("routing map read in descending expert order",
     "for (int e = 0; e < E; ++e) {\n            if (!routing_map[t * E + e]) continue;",
     "for (int e = E - 1; e >= 0; --e) {\n            if (!routing_map[t * E + e]) continue;", 0),
    ("non-expand row for every slot of a rank", "if (ej >= 0 && ej < E && ej / L == r) { first = 0; break; }",
     "if (0) { first = 0; break; }", 0),
    ("alignment pads exact multiples", "run += (c + A - 1) / A * A;", "run += (c + A) / A * A;", 0),
    ("e4m3 saturates to NaN", "if (a >= 448.0) return (uint8_t)(sign | 0x7E);",
     "if (a >= 448.0) return (uint8_t)(sign | 0x7F);", 0),
    ("e5m2 saturates to infinity", "if (a >= 57344.0) return (uint8_t)(sign | 0x7B);",
     "if (a >= 57344.0) return (uint8_t)(sign | 0x7C);", 0),
    ("zero block gets scale 1", "srow[b] = 0.0f;", "srow[b] = 1.0f;", 0),
    ("source token is the slot index", "if (recv_src_token) recv_src_token[row] = (int32_t)t;",
     "if (recv_src_token) recv_src_token[row] = (int32_t)k;", 0),
    ("missing weights read as zero", "float wk = w ? w[k] : 1.0f;", "float wk = w ? w[k] : 0.0f;", 0),
    ("invalid expert id not reported", "if (e < -1 || e >= E) { status = ORC_ERR_EXPERT; continue; }",
     "if (e < -1 || e >= E) { continue; }", 0),
    ("routing map without probs gives zero weights",
     "topk_weights[t * K + k] = probs ? probs[t * E + e] : 1.0f;",
     "topk_weights[t * K + k] = probs ? probs[t * E + e] : 0.0f;", 0),
    ("strided capacity off by one", "if (rank_in_expert >= cap) {", "if (rank_in_expert > cap) {", 0),
    ("strided overflow not reported", "if (status == ORC_OK) status = ORC_ERR_CAPACITY;", ";", 0),
    ("pad rows keep source 0", "if (src) src[r] = -1;", "if (src) src[r] = 0;", 0),
    ("pad rows half zeroed", "memset(recv + r * row_bytes, 0, (size_t)row_bytes);",
     "memset(recv + r * row_bytes, 0, (size_t)row_bytes / 2);", 0),
    ("probs keep the last weight instead of the sum", "probs[t * E + e] += w[t * K + k];",
     "probs[t * E + e] = w[t * K + k];", 0),
    ("non-expand rank offsets inclusive",
     "for (int r = 0; r < R; ++r) { rank_offsets[r] = (int32_t)run; run += num_tokens_per_rank[r]; }",
     "for (int r = 0; r < R; ++r) { run += num_tokens_per_rank[r]; rank_offsets[r] = (int32_t)run; }", 0),
    ("dropped slot gets weight gradient 1",
     "grad_topk_weights[s] = row >= 0 ? grad_recv_weights[row] : 0.0f;",
     "grad_topk_weights[s] = row >= 0 ? grad_recv_weights[row] : 1.0f;", 0),
    ("e4m3 dispatch scales at the token's row",
     "memcpy(recv_scales + (int64_t)row * nb, s, (size_t)nb * sizeof(float));",
     "memcpy(recv_scales + t * nb, s, (size_t)nb * sizeof(float));", 0),
    ("e4m3 dispatch codes at the token's row", "memcpy(recv_q + (int64_t)row * H, q, (size_t)H);",
     "memcpy(recv_q + t * H, q, (size_t)H);", 0),
    ("e4m3 dispatch weight of the next slot",
     "if (recv_weights && topk_weights) recv_weights[row] = topk_weights[t * K + k];",
     "if (recv_weights && topk_weights) recv_weights[row] = topk_weights[t * K + (k + 1) % K];", 1),
    ("bf16 dispatch weight of the next slot",
     "if (recv_weights && topk_weights) recv_weights[row] = topk_weights[t * K + k];",
     "if (recv_weights && topk_weights) recv_weights[row] = topk_weights[t * K + (k + 1) % K];", 0),
    ("non-expand weight of the row's slot for every entry", "on && w ? w[t * K + j] : 0.0f;",
     "on && w ? w[t * K + k] : 0.0f;", 0),
    ("non-expand weight kept on an off-rank slot", "on && w ? w[t * K + j] : 0.0f;", "w ? w[t * K + j] : 0.0f;", 0),
    ("non-expand ids left global", "recv_topk_idx[(int64_t)row * K + j] = on ? ej - r * L : -1;",
     "recv_topk_idx[(int64_t)row * K + j] = on ? ej : -1;", 0),
    ("row permute reads the row index as the token",
     "if (row >= 0) memcpy(recv + (int64_t)row * row_bytes, src + t * row_bytes, (size_t)row_bytes);",
     "if (row >= 0) memcpy(recv + (int64_t)row * row_bytes, src + (row % T) * row_bytes, (size_t)row_bytes);", 0),
    ("strided offsets one block late", "for (int e = 0; e <= E; ++e) expert_offsets[e] = e * cap;",
     "for (int e = 0; e <= E; ++e) expert_offsets[e] = (e + 1) * cap;", 0),
    ("strided rows from the packed offset", "row_of_slot[s] = (int32_t)(e * cap) + rank_in_expert;",
     "row_of_slot[s] = packed[e] + rank_in_expert;", 0),
]


def _mutate(text, old, new, occurrence):
    at = -1
    for _ in range(occurrence + 1):
        at = text.index(old, at + 1)
    return text[:at] + new + text[at + len(old):]


def _run_pins(lib):
    env = dict(os.environ, ORACLE_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, (r.stdout + r.stderr)[-600:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    src = open(SRC).read()
    d = tmp_path_factory.mktemp("mutants")
    jobs = [("unmodified", src)] + [(name, _mutate(src, old, new, occ)) for name, old, new, occ in MUTATIONS]

    def one(job):
        i, (name, text) = job
        c, so = str(d / f"m{i}.c"), str(d / f"m{i}.so")
        open(c, "w").write(text)
        subprocess.run(oracle.compile_command(c, so), check=True)
        return name, _run_pins(so)

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        return dict(ex.map(one, enumerate(jobs)))


def test_mutations_apply_to_the_source():
    src = open(SRC).read()
    for name, old, new, occ in MUTATIONS:
        assert src.count(old) > occ, name


def test_unmodified_copy_passes_every_pin(outcomes):
    code, tail = outcomes["unmodified"]
    assert code == 0, tail


@pytest.mark.parametrize("name", [m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(outcomes, name):
    code, tail = outcomes[name]
    assert code == 1, f"no pin caught: {name}\n{tail}"
