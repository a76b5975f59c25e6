"""The oracle's pins catch plausible mistakes.  Each case plants one mistake
in a copy of rope_chain_oracle.c (an exact text substitution, so the case
fails loudly if the source no longer holds the line), builds it with the
oracle's own flags, and runs the pin tests against it: at least one must
fail (or the run must crash, for a mistake that writes out of bounds).
The unmodified copy, built the same way, must pass them all."""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = ["tests/test_oracle_bf16.py", "tests/test_oracle_norms.py",
        "tests/test_oracle_project_store.py", "tests/test_oracle_variants.py",
        "tests/test_oracle_qkv_front.py"]

MUTANTS = [
    ("hidden norm output not rounded to bf16",
     "            z[c] = rco_f32(rco_bf16_rn(y));\n",
     "            z[c] = y;\n"),
    ("8192-wide sum: warp sums added right to left",
     "    float s = butterfly32(&lane[0]);\n    for (int w = 1; w < 8; ++w) {\n",
     "    float s = butterfly32(&lane[224]);\n    for (int w = 6; w >= 0; --w) {\n"),
    ("8192-wide sum: in-thread order (i, k) instead of (k, i)",
     "        for (int k = 0; k < 4; ++k)\n            for (int i = 0; i < 8; ++i) {\n",
     "        for (int i = 0; i < 8; ++i)\n            for (int k = 0; k < 4; ++k) {\n"),
    ("K-norm mean over 128 instead of 64",
     "    const float inv_hd = 1.0f / 64.0f;   /* exact: 2^-6 */\n",
     "    const float inv_hd = 1.0f / 128.0f;\n"),
    ("64-wide sum: even and odd squares added pairwise first",
     "        ev[j] = k[2 * j] * k[2 * j];\n        od[j] = k[2 * j + 1] * k[2 * j + 1];\n",
     "        ev[j] = k[2 * j] * k[2 * j] + k[2 * j + 1] * k[2 * j + 1];\n        od[j] = 0.0f;\n"),
    ("RoPE: wrong sign on the first output",
     "    *xo = fmaf(x, c, -ys);\n",
     "    *xo = fmaf(x, c, ys);\n"),
    ("store: cos and sin columns swapped",
     "                        float c = rco_f32(cos_sin[pos * RCO_HEAD + j]);\n"
     "                        float sn = rco_f32(cos_sin[pos * RCO_HEAD + RCO_HEAD / 2 + j]);\n",
     "                        float c = rco_f32(cos_sin[pos * RCO_HEAD + RCO_HEAD / 2 + j]);\n"
     "                        float sn = rco_f32(cos_sin[pos * RCO_HEAD + j]);\n"),
    ("store: V half of the cache written from K",
     "memcpy(dst + RCO_HEAD, vh,", "memcpy(dst + RCO_HEAD, kh,"),
    ("store: block and page of a slot swapped",
     "            int64_t blk = s / block_size, page = s % block_size;\n",
     "            int64_t page = s / block_size, blk = s % block_size;\n"),
    ("inverse RMS without eps",
     "    float v = fmaf(sumsq, inv_width, eps);\n",
     "    float v = sumsq * inv_width;\n"),
    ("bf16 rounding: ties away from zero instead of to even",
     "    u += 0x7FFFu + ((u >> 16) & 1u);\n",
     "    u += 0x8000u;\n"),
    ("layer norms: gains not applied",
     "                float y = z[c] * r2;\n                if (g)\n                    y = y * rco_f32(g[c]);\n",
     "                float y = z[c] * r2;\n"),
    ("norm options: gain center not added",
     "    if (n->center != 0.0f)\n        g = g + n->center;\n",
     "    (void)n->center;\n"),
    ("norm options: input-scale weight applied after the sum of squares",
     "        u[c] = pre_scale ? norm_gain(n, offset, c) * v[c] : v[c];\n",
     "        u[c] = v[c];\n"),
    ("norm options: FP32 weights read as bf16",
     "    if (n->fp32)\n        g = ((const float *)n->weight)[offset + c];\n",
     "    if (n->fp32)\n        g = rco_f32(rco_bf16_rn(((const float *)n->weight)[offset + c]));\n"),
    ("projection: every layer uses layer 0's W",
     "                const uint16_t *w = W + (int64_t)l * D * N;\n",
     "                const uint16_t *w = W;\n"),
    ("projection: W [L, N, D] read as [L, D, N]",
     "                        double p = (double)rco_f32(a[k]) * (double)rco_f32(wn[k]);\n",
     "                        double p = (double)rco_f32(a[k]) * (double)rco_f32(w[(int64_t)k * N + n]);\n"),
    ("store: RoPE at the row index instead of the row's position",
     "                pos = positions[t];\n",
     "                pos = t;\n"),
    ("store: a slot past the cache skipped without being counted",
     "            if (s >= capacity) {\n                skipped += 1;\n",
     "            if (s >= capacity) {\n"),
    ("store: K heads addressed with V's row stride",
     "                const uint16_t *kh = k + l * k_layer_stride + t * k_row_stride + (int64_t)h * RCO_HEAD;\n",
     "                const uint16_t *kh = k + l * k_layer_stride + t * v_row_stride + (int64_t)h * RCO_HEAD;\n"),
    ("QKV front: Q heads passed through without the QK-norm",
     "        for (int32_t h = 0; h < num_heads + num_kv_heads; ++h) {\n",
     "        memcpy(o, rr, (size_t)q_size * sizeof(uint16_t));\n"
     "        for (int32_t h = num_heads; h < num_heads + num_kv_heads; ++h) {\n"),
    ("QKV front: a bad position still inserted",
     "        const int insert = s >= 0 && !bad_slot && !bad_pos;\n",
     "        const int insert = s >= 0 && !bad_slot;\n"),
    ("layer norms: every layer takes layer 0's gains",
     "            const uint16_t *g = pre_w ? pre_w + (int64_t)l * RCO_D : NULL;\n",
     "            const uint16_t *g = pre_w ? pre_w : NULL;\n"),
    ("hidden norm: gain applied before the inverse RMS is rounded in",
     "            float y = v[c] * r;\n            if (hidden_w)\n                y = y * rco_f32(hidden_w[c]);\n",
     "            float y = v[c];\n            if (hidden_w)\n                y = y * rco_f32(hidden_w[c]);\n            y = y * r;\n"),
    ("inverse RMS: eps added after the square root",
     "    float v = fmaf(sumsq, inv_width, eps);\n    float root = sqrtf(v);\n",
     "    float v = sumsq * inv_width;\n    float root = sqrtf(v) + eps;\n"),
    ("RoPE: rounded products instead of the fused multiply-adds",
     "    *xo = fmaf(x, c, -ys);\n",
     "    *xo = x * c - ys;\n"),
    ("float64 to bf16: rounded through binary32 first",
     "    if (isnan(d))\n        return (uint16_t)0x7FFFu;\n    uint16_t sign",
     "    if (isnan(d))\n        return (uint16_t)0x7FFFu;\n    if (d == d)\n        return rco_bf16_rn((float)d);\n    uint16_t sign"),
    ("store: a negative slot counted as an error",
     "            if (s < 0)\n                continue;\n            if (s >= capacity) {",
     "            if (s < 0) {\n                skipped += 1;\n                continue;\n            }\n            if (s >= capacity) {"),
    ("QKV front: the gate columns dropped",
     "(size_t)(kv_size + q_size) * sizeof(uint16_t));",
     "(size_t)(kv_size) * sizeof(uint16_t));"),
    ("norm options: the layer norms read the hidden norm's options",
     "            norm_row(z, pre, (int64_t)l * RCO_D, y);\n",
     "            norm_row(z, hidden, 0, y);\n"),
    ("norm options: the layer norm reads the unrounded hidden output",
     "        for (int c = 0; c < RCO_D; ++c)\n            z[c] = rco_f32(rco_bf16_rn(y[c]));\n",
     "        for (int c = 0; c < RCO_D; ++c)\n            z[c] = y[c];\n"),
    ("bf16 rounding: subnormal results flushed to zero",
     "    u += 0x7FFFu + ((u >> 16) & 1u);\n",
     "    if ((u & 0x7F800000u) == 0u)\n        u &= 0x80000000u;\n    u += 0x7FFFu + ((u >> 16) & 1u);\n"),
    ("QKV front: only the K heads rotated",
     "                if (rotate) {\n",
     "                if (rotate && h >= num_heads) {\n"),
    ("QKV front: a bad row counted once per problem",
     "        if ((bad_pos || bad_slot) && err)\n            *err += 1;\n",
     "        if (err)\n            *err += bad_pos + bad_slot;\n"),
    ("projection: the magnitude bound sums signed products",
     "                        if (ab)\n                            ab[n] = ab[n] + fabs(p);\n",
     "                        if (ab)\n                            ab[n] = ab[n] + p;\n"),
    ("projection: the selected rows ignored",
     "            int64_t t = rows ? rows[i] : i;\n",
     "            int64_t t = i;\n"),
    ("bf16 rounding: NaN to 0x7FC0 instead of the box's canonical NaN",
     "    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)\n        return (uint16_t)0x7FFFu;\n",
     "    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)\n        return (uint16_t)0x7FC0u;\n"),
    ("layer norms: the sum of squares taken over x instead of the hidden output",
     "            float r2 = rco_inv_rms(rco_row_sumsq(z), inv_d, eps);\n",
     "            float r2 = rco_inv_rms(rco_row_sumsq(v), inv_d, eps);\n"),
    ("projection: every layer reads layer 0's normed rows",
     "            const uint16_t *a = normed + ((int64_t)l * T + t) * D;\n",
     "            const uint16_t *a = normed + t * D;\n"),
    ("store: NeoX pairs (j, j + 32) instead of GPT-J pairs (2j, 2j + 1)",
     "                    float y0 = kf[2 * j] * r;\n"
     "                    float y1 = kf[2 * j + 1] * r;\n",
     "                    float y0 = kf[j] * r;\n"
     "                    float y1 = kf[j + RCO_HEAD / 2] * r;\n"),
    ("norm options: a gain centre of 0 still added (-0.0 weights become +0.0)",
     "    if (n->center != 0.0f)\n        g = g + n->center;\n",
     "    g = g + n->center;\n"),
    ("float64 to bf16: subnormals rounded at binary32's spacing",
     "    if (qe < -133)\n        qe = -133;                   /* subnormal spacing 2^-133 */\n",
     "    if (qe < -149)\n        qe = -149;\n"),
    ("QKV front: a negative slot counted as an error",
     "        const int bad_slot = s >= capacity;\n",
     "        const int bad_slot = s >= capacity || (slots && s < 0);\n"),
    ("QKV front: cached K taken from the raw projection",
     "                memcpy(dst, o + q_size + h * RCO_HEAD,",
     "                memcpy(dst, rr + q_size + h * RCO_HEAD,"),
    ("QKV front: cached K taken from the Q heads",
     "                memcpy(dst, o + q_size + h * RCO_HEAD,",
     "                memcpy(dst, o + h * RCO_HEAD,"),
]


def _run_pins(tmp_path, old, new):
    src = open(oracle._SRC).read()
    if old is not None:
        assert src.count(old) == 1, "the line to mutate is no longer in the oracle"
        src = src.replace(old, new)
    c_file = tmp_path / "mutant.c"
    c_file.write_text(src)
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(so), str(c_file), "-lm"], check=True)
    env = dict(os.environ, RCO_ORACLE_LIB=str(so))
    return subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "not gpu",
                           "-p", "no:cacheprovider", *PINS],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_unmodified_copy_passes_the_pins(tmp_path):
    r = _run_pins(tmp_path, None, None)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    r = _run_pins(tmp_path, old, new)
    # 1: a pin failed; a negative code: the planted mistake crashed the run
    # (an address mistake can write outside the cache).  Collection or
    # usage errors (2-5) do not count as caught.
    assert r.returncode == 1 or r.returncode < 0, \
        f"no pin failed with the mistake '{name}' planted (exit {r.returncode}):\n{r.stdout[-1500:]}"
