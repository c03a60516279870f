"""Planted mistakes: each pin must reject a plausible error in the oracle.

The oracle is built once per mistake with ORC_MUTANT=n (the list is in
oracle/sd_oracle.c: a dropped term, a wrong sign, a swapped operand or index,
a wrong order), every oracle call is routed to that build, and the pins that
cover the mistake's place are run: at least one of them must fail.  A pin set
that still passes would let that mistake through, and the CUDA path's parity
against the oracle would prove nothing there.  Everything runs on the CPU.
"""

import pytest

import oracle
from tests import test_oracle_ladder as ol
from tests import test_oracle_model as om
from tests import test_oracle_ops as oo

KQ8, KQ4, KA8 = 1, 2, 3

MUTANTS = {
    1: ("fp16 rounding truncates", [oo.test_fp16_conversions_match_numpy]),
    2: ("Q4_0 nibble halves swapped", [oo.test_q4_0_hand_block]),
    3: ("Q8_0 codes read unsigned", [oo.test_q8_0_hand_block]),
    4: ("affine group bias dropped", [oo.test_a8g64_hand_group]),
    5: ("linear layer bias dropped", [lambda: oo.test_linear_against_float64_dot(KQ8)]),
    6: ("LayerNorm unbiased variance", [oo.test_layernorm_invariants_and_torch]),
    7: ("RMSNorm gain dropped", [oo.test_rmsnorm_invariants_and_torch]),
    8: ("GELU with erf instead of the tanh form", [oo.test_activations_against_torch]),
    9: ("RoPE rotates the wrong way", [oo.test_rope_identity_norms_and_complex_form]),
    10: ("attention scores unscaled", [oo.test_attention_closed_forms_and_sdpa]),
    11: ("attention misses the newest key", [om.test_tiny_gpt2_incremental_equals_full_recompute]),
    12: ("sampler drops top-k ties", [oo.test_sampler_adversarial_ties_and_boundaries]),
    13: ("top-p cut one element late", [oo.test_sampler_bruteforce_random_logits]),
    14: ("draw in probability order", [oo.test_sampler_bruteforce_random_logits]),
    15: ("temperature multiplies", [oo.test_sampler_bruteforce_random_logits]),
    16: ("attention residual dropped", [om.test_tiny_gpt2_incremental_equals_full_recompute]),
    17: ("SwiGLU gate and up swapped", [om.test_llama_gqa_rows_match_full_recompute]),
    18: ("query heads interleaved over KV heads", [om.test_llama_gqa_rows_match_full_recompute]),
    19: ("RoPE skipped on keys", [om.test_llama_gqa_rows_match_full_recompute]),
    20: ("repetition penalty backwards", [ol.test_repetition_penalty_divides_positive_and_multiplies_negative_logits]),
    21: ("ladder: top-k before top-p", [ol.test_top_p_acts_before_top_k]),
    22: ("margin ignores membership flips", [oo.test_sampler_margin_at_a_top_k_boundary,
                                             oo.test_sampler_margin_bruteforce_changes_below_it_keep_the_token]),
    23: ("margin taken as if T were 1", [oo.test_sampler_margin_at_a_top_k_boundary]),
    24: ("top-p bound counts an entry before itself", [oo.test_sampler_margin_is_the_draw_distance_when_no_flip_reaches,
                                                       oo.test_sampler_margin_at_a_top_p_cut_that_can_shrink]),
    25: ("mass factor 1+r instead of its square root", [oo.test_sampler_margin_at_a_top_p_cut_that_can_shrink,
                                                         oo.test_sampler_margin_at_a_top_p_cut_that_can_grow]),
    26: ("Q5_0 fifth bit taken from the wrong element", [oo.test_q5_0_hand_block]),
    27: ("4-bit affine codes read high nibble first", [lambda: oo.test_a4_hand_group(oo.KA4G32, 32)]),
    28: ("plain sampler's penalty backwards", [oo.test_penalised_sampler_follows_the_sign_rule]),
}


@pytest.mark.parametrize("n", sorted(MUTANTS))
def test_planted_mistake_is_rejected(n):
    what, pins = MUTANTS[n]
    path = oracle.build_mutant(n)
    caught = []
    with oracle.using_library(path):
        for pin in pins:
            try:
                pin()
            except AssertionError as e:
                caught.append(repr(e)[:120])
    assert caught, f"planted mistake {n} ({what}) passed every pin that covers it"


def test_unmutated_build_passes_the_same_pins():
    """The pins used above pass on the oracle itself (so a failure above is the
    planted mistake, not a pin that always fails)."""
    for n in (2, 6, 10, 12, 13, 22, 24, 25):
        for pin in MUTANTS[n][1]:
            pin()
