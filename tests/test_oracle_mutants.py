"""Plant mistakes in a copy of the CPU oracle and check that the pins catch them.

Each mutant is the oracle's C source with one plausible slip (wrong tie rule,
wrong block width, dropped term, wrong sign, wrong index).  It is compiled in
a temporary directory, loaded in place of the real oracle, and every pin is
run; the mutant must fail at least one.  Nothing here touches a GPU.
"""
import shutil

import pytest

import oracle
import pins

# the expert-selection line of each weight-gradient loop, with enough of the
# loop body to make it unique
_DWD_SEG = ("    for (int s = 0; s < num_seg; ++s) {\n      if (seg_expert_of(seg_expert, s) != e) continue;\n"
            "      for (int r = seg_offsets[s]; r < seg_offsets[s + 1]; ++r) {\n        const float* d = dy_perm")
_DWGU_SEG = ("    for (int s = 0; s < num_seg; ++s) {\n      if (seg_expert_of(seg_expert, s) != e) continue;\n"
             "      for (int r = seg_offsets[s]; r < seg_offsets[s + 1]; ++r) {\n        const float* dg = dgu")

MUTANTS = {
    "tie_to_higher_id": ("moe_oracle.c", "logit[e] > logit[best]", "logit[e] >= logit[best]"),
    "logit_block_128": ("moe_oracle.h", "#define ORACLE_LOGIT_BLOCK 256", "#define ORACLE_LOGIT_BLOCK 128"),
    "bias_dropped": ("moe_oracle.c", "logit[e] = logit[e] + bias[e];", "logit[e] = logit[e];"),
    "softmax_sum_slot0": ("moe_oracle.c", "s = s + ex[j];", "s = s + ex[0];"),
    "silu_sign": ("moe_oracle.c", "float silu = g / (1.0f + expf(-g));", "float silu = g / (1.0f + expf(g));"),
    "gate_up_swapped": ("moe_oracle.c", "h[(size_t)r * I + i] = silu * u;",
                        "h[(size_t)r * I + i] = u / (1.0f + expf(-u)) * g;"),
    "dispatch_reverse_stable": ("moe_oracle.c", "int row = offsets[e] + fill[e];",
                                "int row = offsets[e + 1] - 1 - fill[e];"),
    "combine_weight_slot0": ("moe_oracle.c", "acc = acc + topk_w[(size_t)t * k + j] * y_perm[row * H + c];",
                             "acc = acc + topk_w[(size_t)t * k] * y_perm[row * H + c];"),
    "swiglu_bwd_sign": ("moe_oracle.c", "sg * (1.0f + g * (1.0f - sg))", "sg * (1.0f - g * (1.0f - sg))"),
    "down_bwd_transposed": ("moe_oracle.c", "dh[i] = dh[i] + d[n] * widen_bf16(w[i]);",
                            "dh[i] = dh[i] + d[n] * widen_bf16(Wd[((size_t)e * H + (i % H)) * I + (n % I)]);"),
    "dWu_uses_dg": ("moe_oracle.c", "su[(size_t)i * H + c] = su[(size_t)i * H + c] + du[i] * a[c];",
                    "su[(size_t)i * H + c] = su[(size_t)i * H + c] + dg[i] * a[c];"),
    "router_bwd_sign": ("moe_oracle.c", "dl[(size_t)t * k + j] = w[j] * (g[j] - s);",
                        "dl[(size_t)t * k + j] = w[j] * (g[j] + s);"),
    "router_dx_wrong_column": ("moe_oracle.c", "Wr[(size_t)c * E + topk_idx[(size_t)t * k + j]]",
                               "Wr[(size_t)c * E + j]"),
    "accumulate_ignored": ("moe_oracle.c", "if (!accumulate) memset(p, 0, n * sizeof(float));",
                           "memset(p, 0, n * sizeof(float));"),
    "e4m3_ties_away": ("moe_oracle.c", "q = (int)nearbyint(m / ldexp(1.0, e - 3));",
                       "q = (int)round(m / ldexp(1.0, e - 3));"),
    "e4m3_bias_8": ("moe_oracle.c", "v = ldexp(1.0 + m / 8.0, field - 7);", "v = ldexp(1.0 + m / 8.0, field - 8);"),
    "e4m3_no_subnormals": ("moe_oracle.c", "q = (int)nearbyint(m / ldexp(1.0, -9));", "q = 0;"),
    "quant_scale_240": ("moe_oracle.c", "amax > 0.0f ? amax / 448.0f : 1.0f", "amax > 0.0f ? amax / 240.0f : 1.0f"),
    "quant_multiplies": ("moe_oracle.c", "e4m3_code(row[j] / s)", "e4m3_code(row[j] * s)"),
    "fp8_up_uses_gate_scale": ("moe_oracle.c", "Wu_scale[(size_t)e * I + i] * su", "Wg_scale[(size_t)e * I + i] * su"),
    "fp8_down_row_scale_dropped": ("moe_oracle.c", "(double)h_scale[r] * Wd_scale", "(double)h_scale[0] * Wd_scale"),
    "fp8_down_wrong_weight_row": ("moe_oracle.c", "const uint8_t* w = Wdq + ((size_t)e * H + n) * I;",
                                  "const uint8_t* w = Wdq + ((size_t)e * H + (H - 1 - n)) * I;"),
    "dispatch_bwd_drops_slot": ("moe_oracle.c", "for (int j = 0; j < k; ++j)\n        acc = acc + dx_perm",
                                "for (int j = 1; j < k; ++j)\n        acc = acc + dx_perm"),
    # weight gradients over a segment table with several segments per expert
    "dWd_by_segment_id": ("moe_oracle.c", _DWD_SEG, _DWD_SEG.replace("seg_expert_of(seg_expert, s) != e", "s != e")),
    "dWd_first_segment_only": ("moe_oracle.c", _DWD_SEG,
                               "int seen = 0;\n" + _DWD_SEG.replace("!= e) continue;", "!= e || seen++) continue;")),
    "dWgu_by_segment_id": ("moe_oracle.c", _DWGU_SEG, _DWGU_SEG.replace("seg_expert_of(seg_expert, s) != e", "s != e")),
    "dWgu_first_segment_only": ("moe_oracle.c", _DWGU_SEG,
                                "int seen = 0;\n" + _DWGU_SEG.replace("!= e) continue;", "!= e || seen++) continue;")),
}

# mutants that a specific pin exists to catch: it must be among the failures
MUST_FAIL = {name: "pin_segments_backward" for name in
             ("dWd_by_segment_id", "dWd_first_segment_only", "dWgu_by_segment_id", "dWgu_first_segment_only")}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    fname, old, new = MUTANTS[name]
    for f in ("moe_oracle.c", "moe_oracle.h"):
        shutil.copy(oracle._DIR / f, tmp_path / f)
    src = (tmp_path / fname).read_text()
    assert src.count(old) == 1, f"mutation anchor not unique/present: {old!r}"
    (tmp_path / fname).write_text(src.replace(old, new))
    L = oracle.load(oracle.build(src_dir=tmp_path))
    prev = oracle.use(L)
    failed = []
    try:
        for pin in pins.ALL_PINS:
            try:
                pin()
            except (AssertionError, RuntimeError):
                failed.append(pin.__name__)
    finally:
        oracle.use(prev)
    assert failed, f"mutant {name} passed every pin"
    if name in MUST_FAIL:
        assert MUST_FAIL[name] in failed, (name, failed)
