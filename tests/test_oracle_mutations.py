"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of oracle/moe_oracle.c (in a temporary
directory, never in the repository), builds it, and runs the pin tests that
cover that function against the mutant: at least one of them must fail.  The
mistakes are the kind a restatement of the sources could plausibly contain --
a flipped tie-break, a transposed index, a dropped rounding, a swapped
operand.  CPU only."""
import importlib.util
import os
import subprocess
import sys

import pytest

import test_oracle_formats as F
import test_oracle_path as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")


def _calls(fn):
    """fn's parametrized argument sets (or one empty set)."""
    marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
    if not marks:
        return [{}]
    names, values = marks[0].args
    names = [n.strip() for n in names.split(",")]
    return [dict(zip(names, v if isinstance(v, (list, tuple)) else (v,))) for v in values]


def _mutant(tmp_path, edits):
    src = open(SRC).read()
    for old, new in edits:
        assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
        src = src.replace(old, new, 1)
    mut_dir = tmp_path / "oracle_mut"
    mut_dir.mkdir()
    (mut_dir / "moe_oracle.c").write_text(src)
    spec = importlib.util.spec_from_file_location("oracle_mut",
                                                  os.path.join(ROOT, "oracle", "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC = str(mut_dir / "moe_oracle.c")
    mod._LIB_DIR = str(mut_dir / "_build")
    mod._LIB = str(mut_dir / "_build" / "liboracle.so")
    mod.build(force=True)
    return mod


MUTATIONS = [
    ("route tie-break to the higher id",
     "if (best < 0 || l[e] > l[best]) best = e;   /* strict: lower id wins ties */",
     "if (best < 0 || l[e] >= l[best]) best = e;",
     [P.test_route_k1_is_argmax, P.test_route_k_equals_e_is_stable_descending_sort]),
    ("route weights reversed",
     "topk_w[(size_t)g * K + j] = (float)(ex[j] / sum);",
     "topk_w[(size_t)g * K + j] = (float)(ex[K - 1 - j] / sum);",
     [P.test_route_weights_softmax]),
    ("bf16 ties away from zero",
     "if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))",
     "if (lower >= 0x8000u)",
     [F.test_bf16_rne_matches_library_cast, F.test_bf16_rne_ties_and_specials]),
    ("e4m3 overflow to NaN instead of saturating",
     "if (a >= 448.0f) return (uint8_t)(sign | 0x7e);",
     "if (a > 464.0f) return (uint8_t)(sign | 0x7f);",
     [F.test_e4m3_encode_rounding_and_saturation]),
    ("e4m3 decode exponent off by one",
     "else v = ldexpf((float)(8 + man), ex - 7 - 3);",
     "else v = ldexpf((float)(8 + man), ex - 7 - 2);",
     [F.test_e4m3_decode_all_codes_match_library, F.test_e4m3_decode_ocp_table]),
    ("e4m3 subnormal spacing 2^-8",
     "uint32_t m = round_half_even(a * 512.0f);",
     "uint32_t m = round_half_even(a * 256.0f);",
     [F.test_e4m3_encode_matches_library_inside_range, F.test_e4m3_encode_rounding_and_saturation]),
    ("quantise scale and inverse swapped",
     "float s = amax / 448.0f;",
     "float s = 448.0f / amax;",
     [F.test_block_quant_matches_library_ops]),
    ("quantise amax from the first block element only",
     "if (v > amax) amax = v;",
     "if (i == 0) amax = v;",
     [F.test_block_quant_matches_library_ops, F.test_block_quant_error_bound_and_amax_code]),
    ("tokens attributed to the wrong source rank (t mod R)",
     [("counts[topk_idx[g * K + j] * R + s] += 1;", "counts[topk_idx[g * K + j] * R + (t % R)] += 1;"),
      ("int32_t row = cursor[e * R + s]++;", "int32_t row = cursor[e * R + (t % R)]++;")],
     None,
     [P.test_dispatch_matches_library_stable_sort, P.test_dispatch_brute_force_all_routings]),
    ("rows of a segment in descending token order",
     [("for (int i = 0; i < E * R; ++i) cursor[i] = offsets[i];",
       "for (int i = 0; i < E * R; ++i) cursor[i] = offsets[i + 1];"),
      ("int32_t row = cursor[e * R + s]++;", "int32_t row = --cursor[e * R + s];")],
     None,
     [P.test_dispatch_matches_library_stable_sort, P.test_dispatch_brute_force_all_routings]),
    ("expert scale off by one expert",
     "float se = identity ? 1.0f : 1.0f + (float)e / 256.0f;",
     "float se = identity ? 1.0f : 1.0f + (float)(e + 1) / 256.0f;",
     [P.test_expert_scale_matches_library_ops]),
    ("combine weights reversed",
     "acc = fmaf(topk_w[g * K + j], v, acc);",
     "acc = fmaf(topk_w[g * K + (K - 1 - j)], v, acc);",
     [P.test_combine_one_hot_weights_pick_the_row, P.test_combine_fp32_within_error_bound_of_exact]),
    ("group score is the smallest logit",
     "if (l[e] > m) m = l[e];",
     "if (l[e] < m) m = l[e];",
     [P.test_grouped_route_matches_library_sort]),
    ("low-latency regions transposed",
     "int64_t row = ((int64_t)e * R + s) * C + slot;",
     "int64_t row = ((int64_t)s * E + e) * C + slot;",
     [P.test_ll_layout_is_the_ragged_layout_in_fixed_regions]),
    ("group selection keeps the lowest-scoring groups",
     "if (best < 0 || gscore[q] > gscore[best]) best = q;",
     "if (best < 0 || gscore[q] < gscore[best]) best = q;",
     [P.test_grouped_route_matches_library_sort]),
    ("equal group scores go to the higher group id",
     "if (best < 0 || gscore[q] > gscore[best]) best = q;",
     "if (best < 0 || gscore[q] >= gscore[best]) best = q;",
     [P.test_grouped_route_matches_library_sort]),
    ("push return drops the last row of each region",
     "for (int slot = 0; slot < counts[e * R + s]; ++slot) {",
     "for (int slot = 0; slot + 1 < counts[e * R + s]; ++slot) {",
     [P.test_ll_push_then_reduce_equals_gather]),
    ("route weights not normalised",
     "topk_w[(size_t)g * K + j] = (float)(ex[j] / sum);",
     "topk_w[(size_t)g * K + j] = (float)(ex[j]);",
     [P.test_route_weights_softmax]),
    ("bf16 truncates instead of rounding",
     "upper += 1u;                                 /* may carry into inf: correct */",
     "upper += 0u;",
     [F.test_bf16_rne_matches_library_cast, F.test_bf16_rne_ties_and_specials]),
    ("partial sums returned without their bf16 rounding",
     "acc = acc + oracle_f32_from_bf16(wire);",
     "acc = acc + part;",
     [P.test_partial_with_one_rank_is_receive_side, P.test_partial_slots_and_error_bound]),
    ("route never marks a chosen expert (the same one picked K times)",
     "chosen[best] = 1;\n            topk_idx[(size_t)g * K + j] = best;\n        }\n        double m",
     "chosen[best] = 0;\n            topk_idx[(size_t)g * K + j] = best;\n        }\n        double m",
     [P.test_route_k_equals_e_is_stable_descending_sort, P.test_route_brute_force_tiny]),
    ("expert offsets read at e instead of e*R",
     "for (int e = 0; e <= E; ++e) expert_offsets[e] = offsets[e * R];",
     "for (int e = 0; e <= E; ++e) expert_offsets[e] = offsets[e];",
     [P.test_dispatch_matches_library_stable_sort]),
    ("inverse quantisation scale as 1/scale instead of 448/amax",
     "float inv = 448.0f / amax;",
     "float inv = 1.0f / s;",
     [F.test_block_quant_matches_library_ops, F.test_block_quant_error_bound_and_amax_code]),
    ("every block of a row keeps the first block's scale",
     "scale[b] = s;",
     "scale[0] = s;",
     [F.test_block_quant_matches_library_ops]),
    ("e4m3 rounding ties up instead of to even",
     "if (frac > 0.5f || (frac == 0.5f && (i & 1u))) i += 1u;",
     "if (frac >= 0.5f) i += 1u;",
     [F.test_e4m3_encode_matches_library_inside_range, F.test_e4m3_encode_rounding_and_saturation]),
    ("FP8 expert stand-in dequantises with the row's first block scale",
     "xhat = oracle_e4m3_decode(q) * recv_scale[(int64_t)row * (H / 128) + h / 128];",
     "xhat = oracle_e4m3_decode(q) * recv_scale[(int64_t)row * (H / 128)];",
     [P.test_expert_scale_matches_library_ops]),
    ("combine gathers the first copy's row for every j",
     "int32_t row = tok2row[g * K + j];\n                float v",
     "int32_t row = tok2row[g * K];\n                float v",
     [P.test_combine_one_hot_weights_pick_the_row, P.test_combine_identity_experts_returns_input]),
    ("combine rounds the running sum to bf16 after every term",
     "acc = fmaf(topk_w[g * K + j], v, acc);",
     "acc = oracle_f32_from_bf16(oracle_bf16_from_f32(fmaf(topk_w[g * K + j], v, acc)));",
     [P.test_combine_fp32_within_error_bound_of_exact]),
    ("FP8 amax floor at 2^-64 (tiny blocks quantise to zero codes)",
     "if (amax < 0x1p-119f) amax = 0x1p-119f;",
     "if (amax < 0x1p-64f) amax = 0x1p-64f;",
     [F.test_block_quant_tiny_blocks_exact]),
    ("FP8 amax floor one binade too high (2^-118)",
     "if (amax < 0x1p-119f) amax = 0x1p-119f;",
     "if (amax < 0x1p-118f) amax = 0x1p-118f;",
     [F.test_block_quant_tiny_blocks_exact]),
    ("partial stored in the slot of the last copy on that rank",
     "if (j0 < 0) j0 = j;",
     "j0 = j;",
     [P.test_partial_slots_and_error_bound]),
]


def _edits(entry):
    _, old, new, _ = entry
    return old if new is None else [(old, new)]


def _run_child(i, tmp):
    """In a child process: build mutant i and run its pins; exit 0 if a pin caught it, 3 if not."""
    import pathlib
    entry = MUTATIONS[i]
    mod = _mutant(pathlib.Path(tmp), _edits(entry))
    for fn in entry[3]:
        for kw in _calls(fn):
            try:
                fn(mod, **kw)
            except AssertionError:
                print(f"caught by {fn.__name__}")
                sys.exit(0)
    sys.exit(3)


@pytest.mark.parametrize("i", range(len(MUTATIONS)), ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(i, tmp_path, oracle):
    # the mutant runs in its own process: a planted mistake may also write out of bounds
    code = (f"import sys; sys.path.insert(0, {os.path.dirname(__file__)!r}); sys.path.insert(0, {ROOT!r}); "
            f"import test_oracle_mutations as M; M._run_child({i}, {str(tmp_path)!r})")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode != 3, f"no pin caught: {MUTATIONS[i][0]}"
    assert r.returncode == 0, f"mutant run failed (rc {r.returncode}): {r.stderr[-2000:]}"


def test_unmutated_oracle_passes_the_same_pins(oracle):
    for entry in MUTATIONS:
        for fn in entry[3]:
            for kw in _calls(fn):
                fn(oracle, **kw)
