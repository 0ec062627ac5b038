"""Plant plausible mistakes in the oracle (CPU only) and check that the pins catch
each one. A pin that still passes with the mistake planted would not be pinning."""
import math

import numpy as np
import pytest

import oracle
import oracle.moe_oracle as om
import test_oracle_pins as pins
import test_oracle_pins_options as pins_opt


def _plant(monkeypatch, name, fn):
    monkeypatch.setattr(om, name, fn)
    monkeypatch.setattr(oracle, name, fn)


def _fails(test, *args):
    with pytest.raises(AssertionError):
        test(*args)


def test_capacity_floor_instead_of_ceil_is_caught(monkeypatch):
    def floor_cap(T, k, N, cf):
        if cf is None or cf <= 0:
            return None
        return int(math.floor(float(np.float32(cf)) * T * k / N))
    _plant(monkeypatch, "capacity", floor_cap)
    _fails(pins.test_capacity_named_workloads_closed_form)


def test_capacity_without_topk_factor_is_caught(monkeypatch):
    def no_k(T, k, N, cf):
        if cf is None or cf <= 0:
            return None
        return int(math.ceil(float(np.float32(cf)) * T / N))
    _plant(monkeypatch, "capacity", no_k)
    _fails(pins.test_capacity_named_workloads_closed_form)


def test_aux_without_division_by_k_is_caught(monkeypatch):
    def aux_no_k(probs, idx, N, k):
        T = idx.shape[0]
        f = om.expert_counts(idx, N) / float(T)
        return float(N * np.sum(f * probs.mean(axis=0)))
    _plant(monkeypatch, "aux_loss", aux_no_k)
    _fails(pins.test_aux_is_one_for_a_zero_router, 8, 2)


def test_aux_after_capacity_is_caught(monkeypatch):
    real_route = om.route

    def route_post_cap(x, w_router, bias, k, cf, valid_mask=None, reroute=False):
        r = real_route(x, w_router, bias, k, cf, valid_mask, reroute)
        T, N = r["logits"].shape
        if T:
            f = r["kept_counts"] / float(T * k)
            r["aux_loss"] = float(N * np.sum(f * r["probs"].mean(axis=0)))
        return r
    _plant(monkeypatch, "route", route_post_cap)
    _fails(pins.test_aux_uses_counts_before_capacity)


def test_reversed_tie_rule_is_caught(monkeypatch):
    def topk_high_id(logits, k):
        T, N = logits.shape
        ids = np.broadcast_to(np.arange(N), (T, N))
        return np.lexsort((-ids, -logits), axis=-1)[:, :k]
    _plant(monkeypatch, "topk_select", topk_high_id)
    _fails(pins.test_topk_brute_force_with_ties)


def test_gate_softmax_over_all_experts_is_caught(monkeypatch):
    def gate_all(logits, idx):
        p = om.full_softmax(logits)
        return np.take_along_axis(p, idx, axis=1)
    _plant(monkeypatch, "gate_weights", gate_all)
    _fails(pins.test_gate_weights_sum_to_one_and_equal_renormalised_probs)


def test_swapped_w1_w3_is_caught(monkeypatch):
    real = om.swiglu_expert
    _plant(monkeypatch, "swiglu_expert", lambda x, w1, w3, w2: real(x, w3, w1, w2))
    _fails(pins.test_swiglu_orientation_with_one_hot_weights)


def test_silu_sign_error_is_caught(monkeypatch):
    _plant(monkeypatch, "silu", lambda z: z / (1.0 + np.exp(z)))
    _fails(pins.test_silu_against_library_sigmoid)


def test_capacity_priority_reversed_is_caught(monkeypatch):
    real = om.capacity_assign

    def latest_first(idx, N, C):
        rank, drop, kept = real(idx[::-1].copy(), N, C)
        return rank[::-1].copy(), drop[::-1].copy(), kept
    _plant(monkeypatch, "capacity_assign", latest_first)
    _fails(pins.test_capacity_invariants, 0.5)


def test_renormalising_after_a_drop_is_caught(monkeypatch):
    real_route = om.route

    def route_renorm(x, w_router, bias, k, cf, valid_mask=None, reroute=False):
        r = real_route(x, w_router, bias, k, cf, valid_mask, reroute)
        w = r["topk_w"] * (1 - r["drop_mask"])
        s = w.sum(axis=1, keepdims=True)
        r["topk_w"] = np.where(s > 0, w / np.where(s > 0, s, 1.0), 0.0)
        return r
    _plant(monkeypatch, "route", route_renorm)
    _fails(pins.test_dropped_slots_give_zero_and_kept_weights_are_not_renormalised)


def test_ignoring_drops_in_the_combine_is_caught(monkeypatch):
    real_route = om.route

    def route_no_drop(x, w_router, bias, k, cf, valid_mask=None, reroute=False):
        r = real_route(x, w_router, bias, k, cf, valid_mask, reroute)
        r["drop_mask"] = np.zeros_like(r["drop_mask"])
        return r
    _plant(monkeypatch, "route", route_no_drop)
    _fails(pins.test_dropped_slots_give_zero_and_kept_weights_are_not_renormalised)


def test_reroute_ignoring_room_is_caught(monkeypatch):
    real = om.reroute_overflow

    def no_room_check(logits, idx, drop, counts, C):
        return real(logits, idx, drop, np.zeros_like(counts), C)
    _plant(monkeypatch, "reroute_overflow", no_room_check)
    _fails(pins_opt.test_reroute_hand_example_k1)


def test_reroute_allowing_own_experts_is_caught(monkeypatch):
    def cand_own(logits_t, idx_t, has_room):
        cand = np.nonzero(has_room)[0]
        return cand[np.lexsort((cand, -logits_t[cand]))]
    monkeypatch.setattr(om, "_reroute_candidates", cand_own)
    _fails(pins_opt.test_reroute_excludes_the_tokens_own_experts)


def test_reroute_latest_first_is_caught(monkeypatch):
    real = om.reroute_overflow

    def reversed_order(logits, idx, drop, counts, C):
        a, b, c, d = real(logits[::-1].copy(), idx[::-1].copy(), drop[::-1].copy(), counts, C)
        return a[::-1].copy(), b[::-1].copy(), c[::-1].copy(), d
    _plant(monkeypatch, "reroute_overflow", reversed_order)
    _fails(pins_opt.test_reroute_hand_example_k1)


# ------------------------------------------------------------- layer options

def test_kl_normalised_by_tokens_only_is_caught(monkeypatch):
    def kl_by_t(idx, N, k):
        T = idx.shape[0]
        if T == 0:
            return 0.0
        f = om.expert_counts(idx, N) / float(T)  # sums to k, not 1
        with np.errstate(divide="ignore"):
            return float(np.sum((1.0 / N) * (np.log(1.0 / N) - np.log(f))))
    _plant(monkeypatch, "aux_kl_uniform", kl_by_t)
    _fails(pins_opt.test_kl_is_zero_for_uniform_routing)


def test_kl_in_the_reverse_direction_is_caught(monkeypatch):
    def kl_reversed(idx, N, k):
        T = idx.shape[0]
        if T == 0:
            return 0.0
        f = om.expert_counts(idx, N) / float(T * k)
        nz = f > 0
        return float(np.sum(f[nz] * (np.log(f[nz]) - np.log(1.0 / N))))  # KL(f || uniform)
    _plant(monkeypatch, "aux_kl_uniform", kl_reversed)
    _fails(pins_opt.test_kl_two_expert_closed_form)


def test_biased_probability_variance_is_caught(monkeypatch):
    _plant(monkeypatch, "aux_prob_variance",
           lambda probs: float(np.var(probs)) if probs.size else 0.0)
    _fails(pins_opt.test_probability_variance_matches_torch_std)


def test_tanh_approximation_of_gelu_is_caught(monkeypatch):
    def gelu_tanh(z):
        return 0.5 * z * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (z + 0.044715 * z ** 3)))
    _plant(monkeypatch, "gelu", gelu_tanh)
    _fails(pins_opt.test_gelu_against_torch_and_the_normal_cdf)


def test_gelu_expert_with_silu_is_caught(monkeypatch):
    def silu_expert(x_rows, w1_e, w2_e):
        xr = np.asarray(x_rows, np.float64)
        return om.silu(xr @ np.asarray(w1_e, np.float64).T) @ np.asarray(w2_e, np.float64).T
    _plant(monkeypatch, "gelu_expert", silu_expert)
    _fails(pins_opt.test_gelu_expert_orientation_and_library)


def test_capacity_counting_padding_tokens_is_caught(monkeypatch):
    # route the whole batch and only then blank the padding rows: padding counts in C
    def route_all_tokens(x, w_router, bias, k, cf, valid, reroute=False):
        r = dict(om.route(x, w_router, bias, k, cf, reroute=reroute))
        pad = ~np.asarray(valid, bool)
        r["topk_idx"] = np.where(pad[:, None], -1, r["topk_idx"])
        r["topk_w"] = np.where(pad[:, None], 0.0, r["topk_w"])
        r["drop_mask"] = np.where(pad[:, None], 1, r["drop_mask"]).astype(np.uint8)
        return r
    monkeypatch.setattr(om, "_route_masked", route_all_tokens)
    _fails(pins_opt.test_capacity_counts_only_valid_tokens)


# ------------------------------------------- near ties of the rerouting proposals

def _near_ties_variant(n_extra=1, use_room=True, exclude_own=True):
    """reroute_near_ties with one step changed: n_extra candidates past the m
    proposals, the room test, or the exclusion of the token's own experts."""
    def fn(logits, idx, drop, counts, C, margin=om.NEAR_TIE_MARGIN):
        out = []
        if C is None:
            return np.zeros(0, dtype=np.int64)
        for t in np.nonzero(drop.any(axis=1))[0]:
            m = int(drop[t].sum())
            allowed = (counts < C) if use_room else np.ones(len(counts), bool)
            allowed = allowed.copy()
            if exclude_own:
                allowed[idx[t]] = False
            cand = np.nonzero(allowed)[0]
            cand = cand[np.lexsort((cand, -logits[t][cand]))]
            v = logits[t][cand[:m + n_extra]]
            if v.size >= 2 and (v[:-1] - v[1:] < margin).any():
                out.append(t)
        return np.asarray(out, dtype=np.int64)
    return fn


def test_near_ties_over_m_candidates_only_is_caught(monkeypatch):
    _plant(monkeypatch, "reroute_near_ties", _near_ties_variant(n_extra=0))
    _fails(pins_opt.test_reroute_near_tie_listed_when_the_best_two_candidates_are_close)


def test_near_ties_over_m_plus_two_candidates_is_caught(monkeypatch):
    _plant(monkeypatch, "reroute_near_ties", _near_ties_variant(n_extra=2))
    _fails(pins_opt.test_reroute_near_tie_looks_at_m_plus_one_candidates_only)


def test_near_ties_ignoring_room_is_caught(monkeypatch):
    _plant(monkeypatch, "reroute_near_ties", _near_ties_variant(use_room=False))
    _fails(pins_opt.test_reroute_near_tie_skips_full_and_own_experts)


def test_near_ties_with_the_tokens_own_experts_is_caught(monkeypatch):
    _plant(monkeypatch, "reroute_near_ties", _near_ties_variant(exclude_own=False))
    _fails(pins_opt.test_reroute_near_tie_skips_full_and_own_experts)


def test_near_ties_variant_with_nothing_changed_passes(monkeypatch):
    # the planted variants differ from the oracle in one step only
    _plant(monkeypatch, "reroute_near_ties", _near_ties_variant())
    pins_opt.test_reroute_near_tie_listed_when_the_best_two_candidates_are_close()
    pins_opt.test_reroute_near_tie_looks_at_m_plus_one_candidates_only()
    pins_opt.test_reroute_near_tie_skips_full_and_own_experts()
    pins_opt.test_reroute_near_ties_are_exactly_the_unstable_proposals()
