"""The oracle's pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle/oracle.c (a dropped
factor, a flipped tie-break, a wrong rounding, a transposed or shifted
index, a swapped operand, a wrong constant or loop bound), builds that copy with the oracle's own flags,
points the oracle module at it, and runs the pins that guard that part: at
least one of them must fail. The real oracle source is never modified; the
planted copy lives in pytest's temporary directory (CPU only).
"""
import os
import shutil
import subprocess

import pytest

import oracle
import test_oracle_pins as pins
from oracle import build as oracle_build

GATE_CASES = pins._load_gate_cases()


def _gate_handworked():
    for case in GATE_CASES:
        pins.test_gate_handworked(case)


def _gate_bruteforce():
    for args in [(8, 4, 2, 2), (16, 4, 2, 3), (12, 3, 2, 4), (16, 8, 3, 5)]:
        pins.test_gate_bruteforce_enumeration(*args)


# the per-token layer's expert loop: a routed slot's expert, then the shared
# experts stored after the E routed ones (the next lines make the site unique)
_SHARED_SITE = ("        const int e = k < K ? ids[k] : E + (k - K);\n"
                "        const uint8_t* We = w13 + (int64_t)e * N13 * H;\n"
                "        for (int n = 0; n < N13; ++n) {\n"
                "          const uint8_t* b = We + (int64_t)n * H;\n"
                "          double acc = 0.0;\n"
                "          for (int hh = 0; hh < H; ++hh) acc += a[hh] * g_e4m3_lut[b[hh]];")

# (name, text in oracle.c, planted replacement, pins expected to catch it)
MUTATIONS = [
    ("renormalised weights lose routed_scaling_factor",
     "      for (int k = 0; k < K; ++k) w[k] = (s[ids[k]] / S) * rsf;",
     "      for (int k = 0; k < K; ++k) w[k] = (s[ids[k]] / S);",
     [_gate_handworked, pins.test_gate_weight_sum_is_rsf_and_linear]),
    ("ties go to the higher index",
     "  return (a->idx < b->idx) ? -1 : (a->idx > b->idx ? 1 : 0);",
     "  return (a->idx > b->idx) ? -1 : (a->idx < b->idx ? 1 : 0);",
     [_gate_handworked, _gate_bruteforce]),
    ("group score from the best expert only",
     "      gkv[g].key = (gsz >= 2) ? (b1 + b2) : b1;",
     "      gkv[g].key = b1;",
     [_gate_handworked, _gate_bruteforce]),
    ("weights from the bias-corrected score",
     "      s[e] = oracle_sigmoid32(l[e]);",
     "      s[e] = oracle_sigmoid32(l[e]) + (bias ? bias[e] : 0.0f);",
     [_gate_handworked, _gate_bruteforce]),
    ("exp with a wrong 1/6! coefficient",
     "  p = fmaf(p, r, 0x1.6c16c2p-10f);  /* 1/6! */",
     "  p = fmaf(p, r, 0x1.6c16c2p-9f);  /* 1/6! */",
     [pins.test_exp32_within_two_ulp, pins.test_sigmoid32_within_three_ulp]),
    ("FP8 ties rounded away from zero",
     "  float u = ldexpf(a, 3 - E);\n  int m = (int)rintf(u);",
     "  float u = ldexpf(a, 3 - E);\n  int m = (int)roundf(u);",
     [pins.test_e4m3_encode_specials_and_torch, pins.test_e4m3_encode_exhaustive_nearest_even]),
    ("FP8 overflow to NaN instead of saturation",
     "  if (a >= 448.0f) return (uint8_t)(sign | 0x7E);",
     "  if (a >= 448.0f) return (uint8_t)(sign | 0x7F);",
     [pins.test_e4m3_encode_specials_and_torch]),
    ("bf16 by truncation",
     "  b += 0x7FFFu + lsb;",
     "  b += 0u * lsb;",
     [pins.test_bf16_round_single_rounding]),
    ("unstable order within an expert",
     "    src2dst[i] = offsets[e] + fill[e];",
     "    src2dst[i] = offsets[e + 1] - 1 - fill[e];",
     [lambda: pins.test_route_invariants(37, 8, 2, False), pins.test_permute_quant_scatter]),
    ("weight scale read with the row index",
     "        c[n] = acc * (double)scale_a[r] * (double)scale_b[(int64_t)e * N + n];",
     "        c[n] = acc * (double)scale_a[r] * (double)scale_b[(int64_t)e * N + (r % N)];",
     [pins.test_grouped_gemm_scales_per_row_and_channel]),
    ("gate and up halves swapped",
     "      double g = C[r * 2 * I + j];\n      double u = C[r * 2 * I + I + j];",
     "      double u = C[r * 2 * I + j];\n      double g = C[r * 2 * I + I + j];",
     [pins.test_silu_mul_closed_forms]),
    ("post-reorder uses slot 0's weight for every slot",
     "      double w = (double)topk_w[(int64_t)t * K + k];",
     "      double w = (double)topk_w[(int64_t)t * K];",
     [pins.test_permute_then_unpermute_is_identity]),
    ("shared experts weighted by routed_scaling_factor",
     "        const uint8_t* W2e = w2 + (int64_t)e * H * I;\n        double wk = k < K ? (double)w[k] : 1.0;",
     "        const uint8_t* W2e = w2 + (int64_t)e * H * I;\n"
     "        double wk = k < K ? (double)w[k] : (double)routed_scaling_factor;",
     [lambda: pins.test_layer_shared_experts_add_dense_mlps(1)]),
    ("block amax carried across blocks",
     "    for (int b = 0; b < nb; ++b) {\n      const uint16_t* blk = x + r * C + (int64_t)b * QB;\n"
     "      float amax = 0.0f;",
     "    float amax = 0.0f;\n    for (int b = 0; b < nb; ++b) {\n"
     "      const uint16_t* blk = x + r * C + (int64_t)b * QB;",
     [pins.test_block_quant_is_row_quant_per_block]),
    ("block weight scale index transposed",
     "          acc += part * (double)scale_a[(int64_t)r * KB + kb] *\n"
     "                 (double)sbe[(int64_t)(n / QB) * KB + kb];",
     "          acc += part * (double)scale_a[(int64_t)r * KB + kb] *\n"
     "                 (double)sbe[(int64_t)kb * NBk + (n / QB)];",
     [pins.test_grouped_gemm_block_exact_with_power_of_two_scales,
      pins.test_grouped_gemm_block_with_uniform_scales_is_per_token_gemm]),
    ("per-token scale divided by 488",
     "    float sc = fmaxf(amax, 1e-10f) / 448.0f;\n    scale[r] = sc;",
     "    float sc = fmaxf(amax, 1e-10f) / 488.0f;\n    scale[r] = sc;",
     [pins.test_row_quant_closed_form]),
    ("requant amax of h before its bf16 rounding",
     "          hb[j] = oracle_bf16_round(g / (1.0 + exp(-g)) * u);\n"
     "          float v = fabsf(bf16_to_f32(hb[j]));",
     "          hb[j] = oracle_bf16_round(g / (1.0 + exp(-g)) * u);\n"
     "          float v = (float)fabs(g / (1.0 + exp(-g)) * u);",
     [pins.test_layer_token_path_equals_step_path_and_is_linear_in_rsf,
      pins.test_layer_single_expert_is_dense_fp8_mlp]),
    ("sigmoid(g) * u instead of silu(g) * u",
     "      h[r * I + j] = g / (1.0 + exp(-g)) * u;",
     "      h[r * I + j] = 1.0 / (1.0 + exp(-g)) * u;",
     [pins.test_silu_mul_closed_forms]),
    ("one group more than topk_group kept",
     "    for (int i = 0; i < TG; ++i) allowed[gkv[i].idx] = 1;",
     "    for (int i = 0; i <= TG && i < G; ++i) allowed[gkv[i].idx] = 1;",
     [_gate_handworked, _gate_bruteforce]),
    ("renormalised over every expert instead of the selected ones",
     "      for (int k = 0; k < K; ++k) S = S + s[ids[k]];",
     "      for (int k = 0; k < E; ++k) S = S + s[k];",
     [_gate_handworked, pins.test_gate_weight_sum_is_rsf_and_linear]),
    ("FP8 subnormals decoded one binade low",
     "    v = ldexp((double)m, -9);",
     "    v = ldexp((double)m, -10);",
     [pins.test_e4m3_decode_matches_format_and_torch]),
    ("GEMM without the per-row activation scale",
     "        c[n] = acc * (double)scale_a[r] * (double)scale_b[(int64_t)e * N + n];",
     "        c[n] = acc * (double)scale_b[(int64_t)e * N + n];",
     [pins.test_grouped_gemm_scales_per_row_and_channel]),
    ("GEMM takes the experts' weights in reverse order",
     "      const uint8_t* Be = B + (int64_t)e * N * Kd;\n      for (int n = 0; n < N; ++n) {",
     "      const uint8_t* Be = B + (int64_t)(E - 1 - e) * N * Kd;\n"
     "      for (int n = 0; n < N; ++n) {",
     [pins.test_grouped_gemm_exact_integers]),
    ("sigmoid with the sign of the exponent flipped",
     "  float e = oracle_exp32(-x);",
     "  float e = oracle_exp32(x);",
     [pins.test_sigmoid32_within_three_ulp]),
    ("pre-reorder scatters the next token's scale",
     "      scale_a[d] = sc[t];",
     "      scale_a[d] = sc[(t + 1) % T];",
     [pins.test_permute_quant_scatter]),
    ("softmax renormalised over every expert",
     "      for (int k = 0; k < K; ++k) S = S + oracle_exp32(l[ids[k]] - m);",
     "      for (int e = 0; e < E; ++e) S = S + oracle_exp32(l[e] - m);",
     [_gate_handworked, pins.test_gate_weight_sum_is_rsf_and_linear]),
    ("softmax normaliser misses the last expert",
     "      for (int e = 0; e < E; ++e) Z = Z + oracle_exp32(l[e] - m);",
     "      for (int e = 0; e < E - 1; ++e) Z = Z + oracle_exp32(l[e] - m);",
     [pins.test_gate_no_renormalise]),
    ("unrenormalised weights lose routed_scaling_factor",
     "      for (int k = 0; k < K; ++k) w[k] = s[ids[k]] * rsf;",
     "      for (int k = 0; k < K; ++k) w[k] = s[ids[k]];",
     [pins.test_gate_no_renormalise]),
    ("softmax selects the smallest logits",
     "      kv[e].key = l[e];",
     "      kv[e].key = -l[e];",
     [_gate_handworked, pins.test_gate_weight_sum_is_rsf_and_linear]),
    ("block GEMM uses the first block's activation scale throughout",
     "          acc += part * (double)scale_a[(int64_t)r * KB + kb] *",
     "          acc += part * (double)scale_a[(int64_t)r * KB] *",
     [pins.test_grouped_gemm_block_exact_with_power_of_two_scales]),
    ("block pre-reorder copies only the first block scale",
     "      memcpy(scale_a + d * nb, sc + (int64_t)t * nb, sizeof(float) * (size_t)nb);",
     "      memcpy(scale_a + d * nb, sc + (int64_t)t * nb, sizeof(float));",
     [pins.test_layer_block_token_path_equals_step_path_with_shared_expert]),
    ("block layer picks the w13 weight-scale row modulo instead of by division",
     "            acc += part * (double)sa[kb] * (double)sbe[(int64_t)(n / QB) * KBH + kb];",
     "            acc += part * (double)sa[kb] * (double)sbe[(int64_t)(n % (N13 / QB)) * KBH + kb];",
     [pins.test_layer_block_single_expert_is_dense_block_mlp,
      pins.test_layer_block_token_path_equals_step_path_with_shared_expert]),
    ("block layer requant carries the amax across blocks",
     "        for (int b = 0; b < KBI; ++b) {\n          float amax2 = 0.0f;",
     "        float amax2 = 0.0f;\n        for (int b = 0; b < KBI; ++b) {",
     [pins.test_layer_block_single_expert_is_dense_block_mlp,
      pins.test_layer_block_token_path_equals_step_path_with_shared_expert]),
    ("shared expert taken as the last routed expert",
     _SHARED_SITE, _SHARED_SITE.replace("E + (k - K);", "E + (k - K) - 1;"),
     [lambda: pins.test_layer_shared_experts_add_dense_mlps(1)]),
    ("up rows dequantised with the gate rows' weight scales",
     "          c[n] = acc * (double)sa * (double)s13[(int64_t)e * N13 + n];",
     "          c[n] = acc * (double)sa * (double)s13[(int64_t)e * N13 + (n % I)];",
     [pins.test_layer_single_expert_is_dense_fp8_mlp,
      pins.test_layer_token_path_equals_step_path_and_is_linear_in_rsf]),
    ("each expert's output overwrites the token's sum",
     "          o[cc] += wk * (acc * (double)sa2 * (double)s2[(int64_t)e * H + cc]);",
     "          o[cc] = wk * (acc * (double)sa2 * (double)s2[(int64_t)e * H + cc]);",
     [pins.test_layer_token_path_equals_step_path_and_is_linear_in_rsf]),
    ("expert histogram counted one slot early",
     "  for (int64_t i = 0; i < n; ++i) offsets[topk_ids[i] + 1] += 1;",
     "  for (int64_t i = 0; i < n; ++i) offsets[topk_ids[i]] += 1;",
     # only the routing pin: its destinations reach past M, so a pin that
     # scatters rows through them would write outside the buffer
     [lambda: pins.test_route_invariants(37, 8, 2, False)]),
    ("an expert's rows all land on its first row",
     "    src2dst[i] = offsets[e] + fill[e];",
     "    src2dst[i] = offsets[e];",
     [lambda: pins.test_route_invariants(37, 8, 2, False),
      pins.test_permute_then_unpermute_is_identity]),
    ("post-reorder reads the slot index instead of its permuted row",
     "      const double* d = down + (int64_t)src2dst[(int64_t)t * K + k] * H;",
     "      const double* d = down + ((int64_t)t * K + k) * H;",
     [pins.test_permute_then_unpermute_is_identity]),
    ("E2M1 subnormal ties rounded away from zero",
     "    int m = (int)rintf(a * 2.0f); /* exact scaling */",
     "    int m = (int)roundf(a * 2.0f); /* exact scaling */",
     [pins.test_e2m1_encode_exhaustive_nearest_even]),
    ("E2M1 normal ties rounded away from zero",
     "  float u = ldexpf(a, 1 - E);     /* units of the ulp 2^(E-1): u in [2, 4) */\n"
     "  int m = (int)rintf(u);",
     "  float u = ldexpf(a, 1 - E);     /* units of the ulp 2^(E-1): u in [2, 4) */\n"
     "  int m = (int)roundf(u);",
     [pins.test_e2m1_encode_exhaustive_nearest_even]),
    ("E2M1 saturating to 4",
     "  if (a >= 6.0f) return (uint8_t)(sign | 0x7); /* saturate (also +-inf) */",
     "  if (a >= 6.0f) return (uint8_t)(sign | 0x6); /* saturate (also +-inf) */",
     [pins.test_e2m1_encode_exhaustive_nearest_even]),
    ("NVFP4 block scale from amax / 4",
     "    uint8_t s = oracle_e4m3_encode((amax / 6.0f) / g);",
     "    uint8_t s = oracle_e4m3_encode((amax / 4.0f) / g);",
     [pins.test_nvfp4_quant_closed_form]),
    ("NVFP4 GEMM without the weights' global scale",
     "        c[n] = acc * (double)ga * (double)gb[e];",
     "        c[n] = acc * (double)ga;",
     [pins.test_grouped_gemm_nvfp4_exact_with_power_of_two_scales]),
    ("NVFP4 GEMM weight block scales in reverse K order",
     "                 g_e4m3_lut[sbe[(int64_t)n * KB + kb]];",
     "                 g_e4m3_lut[sbe[(int64_t)n * KB + (KB - 1 - kb)]];",
     [pins.test_grouped_gemm_nvfp4_exact_with_power_of_two_scales]),
    ("NVFP4 layer requantises h with the input's global scale",
     "        nvfp4_quant_row(hb, I, ga2, q2, sa2);",
     "        nvfp4_quant_row(hb, I, ga1, q2, sa2);",
     [pins.test_layer_nvfp4_single_expert_is_dense_nvfp4_mlp]),
    ("NVFP4 layer without w13's global scale",
     "          c[n] = acc * (double)ga1 * (double)g13[e];",
     "          c[n] = acc * (double)ga1;",
     [pins.test_layer_nvfp4_single_expert_is_dense_nvfp4_mlp,
      pins.test_layer_nvfp4_token_path_equals_step_path_with_shared_expert]),
]


@pytest.fixture
def planted(tmp_path, monkeypatch):
    """Builds a copy of the oracle with one text replacement and makes the
    oracle module load it (restored when the test ends)."""

    def plant(old, new):
        src = open(os.path.join(oracle_build.HERE, "oracle.c")).read()
        assert src.count(old) == 1, "the planted site must exist exactly once"
        (tmp_path / "oracle.c").write_text(src.replace(old, new))
        shutil.copy(os.path.join(oracle_build.HERE, "oracle.h"), tmp_path / "oracle.h")
        so = tmp_path / "liboracle_planted.so"
        subprocess.run(["gcc", *oracle_build.CFLAGS, str(tmp_path / "oracle.c"), "-o", str(so),
                        "-lm"], check=True)
        monkeypatch.setattr(oracle_build, "build", lambda force=False: str(so))
        monkeypatch.setattr(oracle, "_lib", None)

    return plant


@pytest.mark.parametrize("name,old,new,guards", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(planted, name, old, new, guards):
    planted(old, new)
    caught = []
    for guard in guards:
        try:
            guard()
        except AssertionError:
            caught.append(getattr(guard, "__name__", "pin"))
    assert caught, f"no pin caught: {name}"
