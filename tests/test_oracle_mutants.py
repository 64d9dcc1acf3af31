"""The oracle's pins catch plausible mistakes.

Each case copies oracle.c, plants one mistake in the copy (a wrong loop order,
mul+add for an FMA, ties away from zero, a reversed slot loop, a wrong sign,
a wrong index, a wrong padding rule ...), builds it, routes the oracle to the
mutant and runs the pins that guard that part: at least one must fail.  The
mistakes stay inside the array bounds, so a mutant can only compute wrong
values.  oracle.c itself is never modified.
"""
from __future__ import annotations

import os
import subprocess

import pytest

import oracle
from tests import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def _brute_map():
    for s in range(12):
        pins.test_build_map_brute_force(s)


def _exact_chain():
    for wp in (True, False):
        for s in range(3):
            pins.test_unpermute_exact_fma_chain(wp, s)


def _sort_pad_brute():
    for s in range(12):
        pins.test_sort_chunks_pad_brute_force(s)


def _capacity_brute():
    for s in range(30):
        pins.test_build_map_capacity_brute_force(s)


def _ep_exact():
    for ep, b, f in ((2, True, False), (4, False, True), (4, True, True), (8, True, False)):
        pins.test_unpermute_ep_exact_tree(ep, b, f)


MUTANTS = {
    "map: slots before tokens inside an expert": (
        """        for (int64_t t = 0; t < T; ++t) {
            for (int32_t k = 0; k < K; ++k) {
                int64_t i = t * K + k;
                if (orc_expert_of(idx, i, E) == e) {
                    row_id_map[i] = next;""",
        """        for (int32_t k = 0; k < K; ++k) {
            for (int64_t t = 0; t < T; ++t) {
                int64_t i = t * K + k;
                if (orc_expert_of(idx, i, E) == e) {
                    row_id_map[i] = next;""",
        [pins.test_worked_example_from_page, _brute_map]),
    "map: rows counted from one": (
        "    int32_t next = 0;\n", "    int32_t next = 1 % (int32_t)(T * K + 1);\n",
        [pins.test_worked_example_from_page, _brute_map]),
    "bf16: ties away from zero": (
        "if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u) != 0u))", "if (lo >= 0x8000u)",
        [pins.test_bf16_rne_against_exact_rounding,
         pins.test_bf16_rne_matches_torch_and_widening_is_exact]),
    "bf16: truncation": (
        "        hi += 1u;\n", "        hi += 0u;\n",
        [pins.test_bf16_rne_against_exact_rounding]),
    "unpermute: multiply then add": (
        "acc = fmaf(probs[t * K + k], r, acc);", "acc = acc + probs[t * K + k] * r;",
        [pins.test_unpermute_fma_differs_from_mul_add, _exact_chain]),
    "unpermute: slots in reverse order": (
        """            float acc = 0.0f;
            for (int32_t k = 0; k < K; ++k) {""",
        """            float acc = 0.0f;
            for (int32_t k = K - 1; k >= 0; --k) {""",
        [_exact_chain, pins.test_unpermute_fma_differs_from_mul_add]),
    "unpermute: probability of the wrong slot": (
        "acc = fmaf(probs[t * K + k], r, acc);", "acc = fmaf(probs[t * K + (k + 1) % K], r, acc);",
        [_exact_chain]),
    "permute: probabilities not permuted": (
        "                out_probs[row] = probs[t * K + k];",
        "                out_probs[row] = probs[t * K];",
        [lambda: pins.test_permute_places_rows_and_probs(False, False)]),
    "permute_bwd: probs gradient read in token order": (
        "g_probs[t * K + k] = row >= 0 ? g_out_probs[row] : 0.0f;",
        "g_probs[t * K + k] = row >= 0 ? g_out_probs[t * K + k] : 0.0f;",
        [pins.test_permute_bwd_is_adjoint_of_permute]),
    "unpermute_bwd: row gradient without the probability": (
        "            float prod = p * g;", "            float prod = g;",
        [pins.test_unpermute_bwd_rows_grad_is_one_rounded_product,
         pins.test_unpermute_bwd_is_adjoint_of_unpermute]),
    "unpermute_bwd: probs gradient with the wrong sign": (
        "                dot += r * (double)g;", "                dot -= r * (double)g;",
        [pins.test_unpermute_bwd_is_adjoint_of_unpermute,
         pins.test_unpermute_bwd_rows_grad_is_one_rounded_product]),
    "sort+pad: a full extra block of padding": (
        "int64_t padded = ((rows_in_group + align - 1) / align) * align;",
        "int64_t padded = (rows_in_group / align + 1) * align;",
        [_sort_pad_brute]),
    "sort+pad: chunk order ignored": (
        """            int32_t c = chunk_order[g * per_group + j];
            if (c < 0 || c >= C) {""",
        """            int32_t c = g * per_group + j;
            if (c < 0 || c >= C) {""",
        [_sort_pad_brute]),
    "capacity: one route too many": (
        "if (capacity < 0 || counts[e] < capacity)", "if (capacity < 0 || counts[e] <= capacity)",
        [_capacity_brute, pins.test_build_map_capacity_keeps_the_earliest_tokens]),
    "EP combine: experts dealt round-robin to ranks": (
        "idx[t * K + k] / per_rank != r", "idx[t * K + k] % ep_size != r",
        [_ep_exact]),
    "EP combine: bf16 partials skipped": (
        """                if (bf16_partials)
                    partial = orc_f32_from_bf16(orc_bf16_from_f32(partial));""",
        """                if (bf16_partials && 0)
                    partial = orc_f32_from_bf16(orc_bf16_from_f32(partial));""",
        [_ep_exact]),
    "fp64 -> bf16: round half up": (
        "double r = rint(a / q) * q;", "double r = floor(a / q + 0.5) * q;",
        [pins.test_bf16_from_f64_against_exact_rounding]),
    "router: ties favour the higher expert": (
        "if (kept[e] && !taken[e] && (best < 0 || l[e] > l[best]))",
        "if (kept[e] && !taken[e] && (best < 0 || l[e] >= l[best]))",
        [pins.test_topk_softmax_selection_matches_stable_argsort]),
    "router: groups scored by their first expert": (
        """                    for (int32_t e = g * per_group + 1; e < (g + 1) * per_group; ++e)
                        if (l[e] > score)
                            score = l[e];""",
        """                    for (int32_t e = g * per_group + 1; e < g * per_group + 1; ++e)
                        if (l[e] > score)
                            score = l[e];""",
        [pins.test_topk_softmax_group_limited_brute_force]),
    "map: rows past the routed ones marked 0 in sorted_to_flat": (
        "            sorted_to_flat[i] = -1;", "            sorted_to_flat[i] = 0;",
        [pins.test_worked_example_from_page, _brute_map, pins.test_build_map_invariants]),
    "sort+pad: padding rows get probability one": (
        "            out_probs[d] = 0.0f;", "            out_probs[d] = 1.0f;",
        [_sort_pad_brute]),
    "unpad+restore backward: padding rows get a gradient": (
        "g_padded[d * H + h] = ok ? g_y[(int64_t)s * H + h] : (uint16_t)0;",
        "g_padded[d * H + h] = ok ? g_y[(int64_t)s * H + h] : (uint16_t)0x3f80;",
        [pins.test_sort_pad_backwards_are_adjoints]),
    "EP combine: fp64 cross-rank sum rounded to fp32 at each rank": (
        "                    acc64 = acc64 + (double)partial;",
        "                    acc64 = (double)(float)(acc64 + (double)partial);",
        [_ep_exact, pins.test_unpermute_ep_fp64_sum_decides_a_bf16_tie]),
    "router backward: sign flipped": (
        "probs[t * K + k] * (g_probs[t * K + k] - d)", "probs[t * K + k] * (d - g_probs[t * K + k])",
        [pins.test_topk_softmax_bwd_is_the_softmax_jacobian]),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_the_planted_mistake(name, tmp_path):
    old, new, checks = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "the mutation no longer applies to oracle.c"
    mutant_c = tmp_path / "oracle_mutant.c"
    mutant_c.write_text(src.replace(old, new, 1))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", *oracle.CFLAGS, str(mutant_c), "-o", str(lib), "-lm"], check=True)
    caught = 0
    with oracle.using_library(str(lib)):
        for check in checks:
            try:
                check()
            except AssertionError:
                caught += 1
    assert caught > 0, f"no pin caught: {name}"


def test_the_unmutated_oracle_passes_the_same_checks():
    for _, _, checks in MUTANTS.values():
        for check in checks:
            check()
