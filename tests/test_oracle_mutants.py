"""Planted mistakes in the oracle: each must fail at least one pin.

The pins of the CPU oracle (brute force, closed forms, invariants, the
worked examples under ``tests/golden/``) are only worth something if a
plausible slip in the oracle's arithmetic breaks one of them.  Each entry
below plants one such slip (a dropped term, a wrong index or sign, an
off-by-one, a transposed operand) in a copy of ``oracle/ep_oracle.c``,
builds that copy, and runs the oracle's pin tests against it
(``EP_ORACLE_SOURCE`` points the ``oracle`` package at the copy).  The
pin suite must fail for every one.  CPU only; nothing here touches a GPU or
the CUDA library.

Slips that stay inside the definitions' own freedom are not planted: for
example an unfused ``acc + w*y`` in the combine differs from the fused form
by less than the combine tolerance, so no pin can (or should) tell them
apart.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
ORACLE_SRC = os.path.join(ROOT, "oracle", "ep_oracle.c")

# the pin suites of the oracle (all CPU)
PIN_FILES = [
    "test_oracle_plan.py",
    "test_oracle_formats.py",
    "test_oracle_dispatch_combine.py",
    "test_oracle_extras.py",
    "test_oracle_backward.py",
    "test_oracle_nonfinite.py",
]

# (name, text in ep_oracle.c (must occur once), replacement)
MUTANTS = [
    # --- number formats ---
    ("bf16 round: ties away from zero",
     "(dropped == 0x8000u && (kept & 1u))", "(dropped == 0x8000u)"),
    ("bf16 round: truncation",
     "        kept += 1u; /* carry", "        kept += 0u; /* carry"),
    ("e4m3 encode: ties away from zero",
     "double r = nearbyint(n);", "double r = floor(n + 0.5);"),
    ("e4m3 encode: no saturation",
     "    if (val > 448.0)\n        val = 448.0; /* satfinite */",
     "    if (val > 480.0)\n        val = 480.0; /* satfinite */"),
    ("e4m3 encode: subnormal spacing 2^-10",
     "        spacing = ldexp(1.0, -9);\n    } else {",
     "        spacing = ldexp(1.0, -10);\n    } else {"),
    ("e4m3 encode: exponent bias 8",
     "int exp_field = (e2 - 1) + 7;", "int exp_field = (e2 - 1) + 8;"),
    ("e4m3 encode: a NaN keeps its sign",
     "        return (uint8_t)0x7f;", "        return (uint8_t)(sign | 0x7f);"),
    ("fp8 amax: a NaN element takes over the group",
     "                if (v > amax)\n                    amax = v;",
     "                if (!(v <= amax))\n                    amax = v;"),
    ("e4m3 encode: infinity to NaN",
     "return (uint8_t)(sign | 0x7e); /* satfinite: +-448 */",
     "return (uint8_t)(sign | 0x7f); /* satfinite: +-448 */"),
    ("e4m3 decode: exponent bias 8",
     "v = ldexp(1.0 + mant / 8.0, exp_field - 7);", "v = ldexp(1.0 + mant / 8.0, exp_field - 8);"),
    ("e4m3 decode: subnormal scale 2^-10",
     "v = ldexp((double)mant, -9); /* subnormal", "v = ldexp((double)mant, -10); /* subnormal"),
    # --- validation ---
    ("validate: duplicate ids accepted",
     "                if (topk_idx[g * K + k2] == e)\n                    return ORACLE_ERR_INVALID;",
     "                if (topk_idx[g * K + k2] == e + E)\n                    return ORACLE_ERR_INVALID;"),
    ("validate: id E accepted",
     "if (e < -1 || e >= E)", "if (e < -1 || e > E)"),
    ("validate: E % P unchecked",
     "if (E % P != 0 || K > E", "if (K > E"),
    # --- plan ---
    ("rank of an expert: e mod P",
     "if (e >= 0 && e / E_l == d)", "if (e >= 0 && e % P == d)"),
    ("per-expert counts: last slot dropped",
     "            for (int64_t t = 0; t < S; ++t)\n                for (int k = 0; k < K; ++k)\n"
     "                    n += topk_idx[((int64_t)s * S + t) * K + k] == e;",
     "            for (int64_t t = 0; t < S; ++t)\n                for (int k = 0; k < K - 1; ++k)\n"
     "                    n += topk_idx[((int64_t)s * S + t) * K + k] == e;"),
    ("rank prefix: exclusive",
     "for (int s2 = 0; s2 <= s; ++s2)", "for (int s2 = 0; s2 < s; ++s2)"),
    ("channel prefix: per channel, not cumulative",
     "                for (int64_t t = lo; t < hi; ++t)\n                    acc += is_token_in_rank",
     "                acc = 0;\n                for (int64_t t = lo; t < hi; ++t)\n"
     "                    acc += is_token_in_rank"),
    ("channel ranges: floor(S/C) tokens",
     "const int64_t chunk = S > 0 ? (S + C - 1) / C : 0;", "const int64_t chunk = S > 0 ? S / C : 0;"),
    ("recv channel prefix: rank prefix transposed",
     "int32_t base = s > 0 ? rank_prefix[(s - 1) * P + d] : 0;",
     "int32_t base = s > 0 ? rank_prefix[d * P + (s - 1)] : 0;"),
    ("recv channel prefix: inclusive channel term",
     "int32_t in_src = c > 0 ? channel_prefix[((int64_t)s * P + d) * C + c - 1] : 0;",
     "int32_t in_src = channel_prefix[((int64_t)s * P + d) * C + c];"),
    ("send_head: global row instead of window row",
     "                send_head[g * P + d] = pos;", "                send_head[g * P + d] = recv_offsets[d] + pos;"),
    ("recv_src_idx: global token instead of source-local",
     "recv_src_idx[recv_offsets[d] + pos] = (int32_t)(g % S);",
     "recv_src_idx[recv_offsets[d] + pos] = (int32_t)g;"),
    ("expert padding: an extra block on exact multiples",
     "((int64_t)expert_counts[e] + A - 1) / A * A", "((int64_t)expert_counts[e] + A) / A * A"),
    ("expert padding: none",
     "int64_t padded = ((int64_t)expert_counts[e] + A - 1) / A * A;",
     "int64_t padded = (int64_t)expert_counts[e] + 0 * A;"),
    ("expanded layout: slot-major order inside a segment",
     "        for (int64_t g = 0; g < T; ++g)\n            for (int k = 0; k < K; ++k)\n"
     "                if (topk_idx[g * K + k] == e) {",
     "        for (int k = 0; k < K; ++k)\n            for (int64_t g = 0; g < T; ++g)\n"
     "                if (topk_idx[g * K + k] == e) {"),
    ("padding rows: exp_src 0 instead of -1",
     "        for (; row < expert_offsets[e + 1]; ++row)\n            exp_src[row] = -1;",
     "        for (; row < expert_offsets[e + 1]; ++row)\n            exp_src[row] = 0;"),
    # --- dispatch ---
    ("bf16 dispatch: padding rows not zeroed",
     "            else if (zero_pad)\n                out[r * H + h] = 0;",
     "            else if (zero_pad)\n                out[r * H + h] = 1;"),
    ("fp8 dispatch: scale by the reciprocal of 448",
     "float scale = amax / 448.0f;", "float scale = amax * (1.0f / 448.0f);"),
    ("fp8 dispatch: signed max instead of amax",
     "                float v = fabsf(ep_oracle_bf16_to_f32(x[(int64_t)g * H + j * 128 + i]));",
     "                float v = ep_oracle_bf16_to_f32(x[(int64_t)g * H + j * 128 + i]);"),
    ("fp8 dispatch: scale 447",
     "float scale = amax / 448.0f;", "float scale = amax / 447.0f;"),
    ("fp8 dispatch: padding scales not zeroed",
     "                    out_scales[r * G + j] = 0.0f;\n            }\n            continue;",
     "                    out_scales[r * G + j] = 1.0f;\n            }\n            continue;"),
    # --- combine ---
    ("combine: bias subtracted",
     "            if (bias)\n                acc = acc + ep_oracle_bf16_to_f32(bias[g * H + h]);",
     "            if (bias)\n                acc = acc - ep_oracle_bf16_to_f32(bias[g * H + h]);"),
    ("combine: last slot dropped",
     "void ep_oracle_combine(const uint16_t *y, int64_t H, const int32_t *slot,\n"
     "                       const float *topk_weights, int64_t T, int K, uint16_t *out)\n{\n"
     "#pragma omp parallel for schedule(static)\n"
     "    for (int64_t g = 0; g < T; ++g)\n        for (int64_t h = 0; h < H; ++h) {\n"
     "            float acc = 0.0f;\n            for (int k = 0; k < K; ++k) {",
     "void ep_oracle_combine(const uint16_t *y, int64_t H, const int32_t *slot,\n"
     "                       const float *topk_weights, int64_t T, int K, uint16_t *out)\n{\n"
     "#pragma omp parallel for schedule(static)\n"
     "    for (int64_t g = 0; g < T; ++g)\n        for (int64_t h = 0; h < H; ++h) {\n"
     "            float acc = 0.0f;\n            for (int k = 0; k < K - 1; ++k) {"),
    ("combine: weights ignored",
     "                acc = fmaf(topk_weights[g * K + k], ep_oracle_bf16_to_f32(y[(int64_t)r * H + h]), acc);\n"
     "            }\n            out[g * H + h]",
     "                acc = fmaf(1.0f, ep_oracle_bf16_to_f32(y[(int64_t)r * H + h]), acc);\n"
     "            }\n            out[g * H + h]"),
    # --- synthetic experts ---
    ("scaling expert: factor 1 + e/(E-1)",
     "        float f = 1.0f + (float)e / (float)E;\n#pragma omp parallel for",
     "        float f = 1.0f + (float)e / (float)(E - 1);\n#pragma omp parallel for"),
    ("dequant expert: scale of the next group",
     "scales[r * G + h / 128]", "scales[r * G + (h / 128 + 1) % G]"),
    # --- backward ---
    ("dispatch backward: only the first slot",
     "                if (r >= 0)\n                    acc = acc + ep_oracle_bf16_to_f32(grad_recv",
     "                if (r >= 0 && k == 0)\n                    acc = acc + ep_oracle_bf16_to_f32(grad_recv"),
    ("combine backward: grad_y without the weight",
     "ep_oracle_f32_to_bf16(wk * go);", "ep_oracle_f32_to_bf16(go);"),
    ("combine backward: grad_w against the token row",
     "dot += (double)go * (double)ep_oracle_bf16_to_f32(y[(int64_t)r * H + h]);",
     "dot += (double)go * (double)ep_oracle_bf16_to_f32(y[(int64_t)g * H + h]);"),
    # --- metadata and pre-quantised input ---
    ("metadata: slot index off by one",
     "            recv_meta[2 * r + 1] = k;", "            recv_meta[2 * r + 1] = k + 1;"),
    ("metadata: weight of slot 0",
     "            recv_weights[r] = topk_weights[g * K + k];", "            recv_weights[r] = topk_weights[g * K];"),
    ("metadata: token off by one",
     "            recv_meta[2 * r] = (int32_t)g;", "            recv_meta[2 * r] = (int32_t)g + 1;"),
    ("combine: bias row of token 0",
     "acc = acc + ep_oracle_bf16_to_f32(bias[g * H + h]);", "acc = acc + ep_oracle_bf16_to_f32(bias[h]);"),
    ("combine backward: padding rows not zeroed",
     "                    grad_y[r * H + h] = 0;", "                    grad_y[r * H + h] = 0x3f80;"),
    ("receive totals: count matrix transposed",
     "            n += num_tokens_per_rank[s * P + d];", "            n += num_tokens_per_rank[d * P + s];"),
    ("recv channel prefix: written [s][d][c]",
     "recv_channel_prefix[((int64_t)d * P + s) * C + c] = base + in_src;",
     "recv_channel_prefix[((int64_t)s * P + d) * C + c] = base + in_src;"),
    ("fp8 input: codes of token 0",
     "out_q[r * H + h] = g >= 0 ? xq[(int64_t)g * H + h] : 0;", "out_q[r * H + h] = g >= 0 ? xq[h] : 0;"),
    ("combine backward: weight gradient on an unused slot",
     "grad_w[g * K + k] = dot;", "grad_w[g * K + k] = r >= 0 ? dot : 1.0;"),
    ("bf16 round: NaN becomes infinity",
     "return (uint16_t)((u >> 16) | 0x0040u);", "return (uint16_t)((u >> 16) & 0xff80u);"),
    ("e4m3 decode: NaN code read as 480",
     "if (exp_field == 0xf && mant == 7)", "if (exp_field == 0xf && mant == 8)"),
    ("validate: channels beyond S accepted",
     "K > E || (S > 0 && C > S)", "K > E || (S > 0 && C > S + 1)"),
    ("worst expanded rows: padding term dropped",
     "return (int64_t)P * S * K + (int64_t)E * (A - 1);", "return (int64_t)P * S * K;"),
    ("worst receive rows: top-k not capped by P",
     "return (int64_t)P * S * (K < P ? K : P);", "return (int64_t)P * S * K;"),
    ("metadata: padding rows weigh 1",
     "        recv_weights[r] = 0.0f;", "        recv_weights[r] = 1.0f;"),
    ("channel ranges: last channel not clipped to S",
     "if (hi > S) hi = S;", "if (hi > S + 1) hi = S + 1;"),
    ("fp8 input: scales of token 0",
     "out_scales[r * G + j] = g >= 0 ? xs[(int64_t)g * G + j] : 0.0f;",
     "out_scales[r * G + j] = g >= 0 ? xs[j] : 0.0f;"),
]


def _mutate(src: str, old: str, new: str) -> str:
    assert src.count(old) == 1, f"mutation site not unique or missing: {old!r}"
    return src.replace(old, new)


def run_mutant(mutant, workdir: str):
    """Builds one mutated oracle in ``workdir`` and runs the pin suite on it.
    Returns (pytest exit code, output tail)."""
    name, old, new = mutant
    with open(ORACLE_SRC) as f:
        src = f.read()
    path = os.path.join(workdir, "ep_oracle_mutant.c")
    with open(path, "w") as f:
        f.write(_mutate(src, old, new))
    # a mutant must still compile: a failing pin then means the pins caught it
    so = os.path.join(workdir, "ep_oracle_mutant.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                    "-o", so, path, "-lm"], check=True, capture_output=True, text=True)
    env = dict(os.environ, EP_ORACLE_SOURCE=path, PYTHONDONTWRITEBYTECODE="1")
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider",
           *[os.path.join(HERE, f) for f in PIN_FILES]]
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return res.returncode, (res.stdout + res.stderr)[-2000:]


def test_mutation_sites_exist():
    with open(ORACLE_SRC) as f:
        src = f.read()
    for name, old, new in MUTANTS:
        assert src.count(old) == 1, name
        assert old != new, name


def test_every_planted_mistake_fails_a_pin():
    survivors = []
    with tempfile.TemporaryDirectory() as tmp:
        def one(i_m):
            i, m = i_m
            d = os.path.join(tmp, str(i))
            os.makedirs(d)
            return m[0], run_mutant(m, d)
        workers = max(1, min(6, (os.cpu_count() or 2) - 1))
        with cf.ThreadPoolExecutor(workers) as ex:
            for name, (rc, out) in ex.map(one, enumerate(MUTANTS)):
                # exit code 1: tests ran and at least one pin failed
                if rc != 1:
                    survivors.append(f"{name} (pytest exit {rc}): {out[-400:]}")
    assert not survivors, "planted mistakes that no pin caught:\n" + "\n".join(survivors)
