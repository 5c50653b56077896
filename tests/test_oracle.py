"""CPU tests of the oracle against its pins, plus planted-mistake checks showing the
pins would catch a plausible error in any one step of the oracle."""

import math

import numpy as np
import pytest

import oracle
import oracle.naive as oa
from tests import oracle_pins as pins


ALL_PINS = pins.ORACLE_PINS + pins.RECURRENCE_PINS + pins.BACKWARD_PINS + pins.GENERAL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oa)


def test_page_facts_are_consistent():
    """The numbers the pages print agree with the mathematics they describe."""
    f = pins.load_page_facts()
    assert math.exp(f["fp16_exp_overflow_arg"]) > f["fp16_max"] > math.exp(f["fp16_exp_overflow_arg"] - 1)
    fp32_max = float(np.finfo(np.float32).max)
    assert math.exp(f["fp32_exp_overflow_near"] - 1) < fp32_max < math.exp(f["fp32_exp_overflow_near"])
    assert abs(math.exp(88) - f["kcs_e88"]) / f["kcs_e88"] < 0.01
    assert abs(2.0 ** 127 - f["kcs_2pow127"]) / f["kcs_2pow127"] < 0.01
    assert abs(math.log2(math.e) - f["log2e"]) < 5e-5


def test_oracle_package_exports():
    for name in ("attention", "attention_rows", "online_softmax_trace", "online_weighted_sum",
                 "attention_backward", "attention_backward_rows", "attention_backward_cols",
                 "attention_general", "merge_partials"):
        assert callable(getattr(oracle, name))


# --------------------------------------------------------------------------- planted mistakes

def _no_scale(q_rows, k, scale):
    return q_rows @ k.T


def _mask_wrong_way(s, rows):
    j = np.arange(s.shape[1])[None, :]
    return np.where(j < rows[:, None], -np.inf, s)


def _mask_drops_diagonal(s, rows):
    j = np.arange(s.shape[1])[None, :]
    return np.where(j >= rows[:, None], -np.inf, s)


def _no_mask(s, rows):
    return s


def _softmax_no_max(s):
    e = np.exp(s)
    l = e.sum(axis=1, keepdims=True)
    return e / l, np.zeros(s.shape[0]), l[:, 0]


def _softmax_unnormalised(s):
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    return e, m[:, 0], e.sum(axis=1)


def _softmax_wrong_axis(s):
    m = s.max(axis=0, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=0, keepdims=True)
    return e / l, s.max(axis=1), np.exp(s - s.max(axis=1, keepdims=True)).sum(axis=1)


def _values_transposed(p, v):
    return p.T @ v


def _lse_base2(m, l):
    return m + np.log2(l)


def _lse_without_max(m, l):
    return np.log(l)


def _trace_no_rescale(x, block):
    m, l, out = -math.inf, 0.0, []
    for s in range(0, len(x), block):
        xb = list(x[s:s + block])
        m = max(m, max(xb))
        l = l + sum(math.exp(t - m) for t in xb)
        out.append((s + len(xb), m, l, 1.0))
    return out


def _weighted_no_acc_rescale(x, vals, block):
    x = np.asarray(x, float)
    vals = np.asarray(vals, float)
    m, l, acc = -np.inf, 0.0, np.zeros(vals.shape[1])
    for s in range(0, len(x), block):
        xb = x[s:s + block]
        m_new = max(m, xb.max())
        a = 0.0 if m == -np.inf else math.exp(m - m_new)
        p = np.exp(xb - m_new)
        l = l * a + p.sum()
        acc = acc + p @ vals[s:s + block]
        m = m_new
    return acc / l, m, l


def _dsoftmax_no_rowsum(p, dp):
    return p * dp


def _dsoftmax_rowsum_of_dp(p, dp):
    return p * (dp - dp.sum(axis=1, keepdims=True))


def _dsoftmax_sign(p, dp):
    return p * (np.sum(p * dp, axis=1, keepdims=True) - dp)


def _dq_no_scale(ds, k, scale):
    return ds @ k


def _dk_no_scale(ds, q_rows, scale):
    return ds.T @ q_rows


def _dp_wrong_operand(do_rows, v):
    return do_rows @ (v[::-1]).T


def _dv_unnormalised(p, do_rows):
    return (p / p.max(axis=1, keepdims=True)).T @ do_rows


def _general_mask_top_left(Tq, Tk, causal, block_mask=None, block=128):
    vis = np.ones((Tq, Tk), dtype=bool)
    if causal:
        vis &= np.arange(Tk)[None, :] <= np.arange(Tq)[:, None]
    if block_mask is not None:
        bm = np.asarray(block_mask) != 0
        vis &= bm[np.arange(Tq) // block][:, np.arange(Tk) // block]
    return vis


def _general_mask_blocks_transposed(Tq, Tk, causal, block_mask=None, block=128):
    vis = np.ones((Tq, Tk), dtype=bool)
    if causal:
        vis &= np.arange(Tk)[None, :] <= (np.arange(Tq) + (Tk - Tq))[:, None]
    if block_mask is not None:
        bm = (np.asarray(block_mask) != 0).T  # block (j, i) looked up for query i, key j
        vis &= bm[np.arange(Tq) // block][:, np.arange(Tk) // block]
    return vis


def _merge_plain_average(o_parts, lse_parts):
    o_parts = np.asarray(o_parts, float)
    return o_parts.mean(axis=0), np.log(np.exp(np.asarray(lse_parts, float)).sum(axis=0))


def _merge_no_shift(o_parts, lse_parts):
    w = np.exp(np.asarray(lse_parts, float))
    o = (w[..., None] * np.asarray(o_parts, float)).sum(axis=0) / w.sum(axis=0)[..., None]
    return o, np.log(w.sum(axis=0))


MUTANTS = {
    "scores:no_scale": ("scores", _no_scale),
    "mask:wrong_direction": ("apply_causal_mask", _mask_wrong_way),
    "mask:drops_diagonal": ("apply_causal_mask", _mask_drops_diagonal),
    "mask:none": ("apply_causal_mask", _no_mask),
    "softmax:no_max_subtraction": ("safe_softmax", _softmax_no_max),
    "softmax:unnormalised": ("safe_softmax", _softmax_unnormalised),
    "softmax:wrong_axis": ("safe_softmax", _softmax_wrong_axis),
    "values:transposed": ("weighted_values", _values_transposed),
    "lse:base2": ("logsumexp_from", _lse_base2),
    "lse:without_max": ("logsumexp_from", _lse_without_max),
    "trace:no_rescale": ("online_softmax_trace", _trace_no_rescale),
    "weighted:no_acc_rescale": ("online_weighted_sum", _weighted_no_acc_rescale),
}

GENERAL_MUTANTS = {
    "general:top_left_causal": ("general_mask", _general_mask_top_left),
    "general:block_mask_transposed": ("general_mask", _general_mask_blocks_transposed),
    "merge:plain_average": ("merge_partials", _merge_plain_average),
    "merge:no_max_shift": ("merge_partials", _merge_no_shift),
}

BACKWARD_MUTANTS = {
    "dsoftmax:no_rowsum": ("softmax_backward", _dsoftmax_no_rowsum),
    "dsoftmax:rowsum_of_dp": ("softmax_backward", _dsoftmax_rowsum_of_dp),
    "dsoftmax:sign": ("softmax_backward", _dsoftmax_sign),
    "dq:no_scale": ("grad_queries", _dq_no_scale),
    "dk:no_scale": ("grad_keys", _dk_no_scale),
    "dp:wrong_operand_order": ("grad_probs", _dp_wrong_operand),
    "dv:unnormalised_p": ("grad_values", _dv_unnormalised),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    attr, broken = MUTANTS[name]
    monkeypatch.setattr(oa, attr, broken)
    failed = pins.run_all(oa, pins.ORACLE_PINS + pins.RECURRENCE_PINS)
    assert failed, f"no pin caught the planted mistake {name}"


@pytest.mark.parametrize("name", sorted(GENERAL_MUTANTS))
def test_general_pins_catch_planted_mistake(name, monkeypatch):
    attr, broken = GENERAL_MUTANTS[name]
    monkeypatch.setattr(oa, attr, broken)
    failed = pins.run_all(oa, pins.GENERAL_PINS)
    assert failed, f"no general-form pin caught the planted mistake {name}"


@pytest.mark.parametrize("name", sorted(BACKWARD_MUTANTS))
def test_backward_pins_catch_planted_mistake(name, monkeypatch):
    attr, broken = BACKWARD_MUTANTS[name]
    monkeypatch.setattr(oa, attr, broken)
    failed = pins.run_all(oa, pins.BACKWARD_PINS)
    assert failed, f"no backward pin caught the planted mistake {name}"


@pytest.mark.parametrize("name", ["scores:no_scale", "mask:drops_diagonal", "mask:none",
                                  "softmax:unnormalised"])
def test_backward_pins_catch_forward_mistake(name, monkeypatch):
    """The backward pins also see a mistake in the shared forward steps."""
    attr, broken = MUTANTS[name]
    monkeypatch.setattr(oa, attr, broken)
    assert pins.run_all(oa, pins.BACKWARD_PINS), name


def test_unmodified_oracle_passes_every_pin():
    assert pins.run_all(oa, ALL_PINS) == []


def test_e4m3_decoding_matches_the_format():
    """The FP8 inputs' decoder (a library cast) against the e4m3 definition: 1 sign bit,
    4 exponent bits with bias 7, 3 mantissa bits; exponent 0 is subnormal (m/8 · 2^-6);
    S.1111.111 is NaN and there is no infinity, so the largest value is 1.75 · 2^8 = 448."""
    import torch
    from exact_attention_23_gb300 import inputs
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    got = inputs.dequantize_e4m3(codes, 1.0)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 0x7
        if e == 0xF and m == 0x7:
            assert np.isnan(got[c]), c
            continue
        want = sign * (m / 8.0 * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7))
        assert got[c] == want, (c, got[c], want)
    assert np.nanmax(got) == inputs.E4M3_MAX


def test_e4m3_quantisation_round_trip():
    """Quantised values are the nearest e4m3 values (relative error ≤ 2^-4) and the scale
    maps the largest magnitude to 448."""
    import torch
    from exact_attention_23_gb300 import inputs
    g = torch.Generator().manual_seed(5)
    x = torch.randn(1000, generator=g) * 3.0
    codes, sc = inputs.quantize_e4m3(x)
    back = inputs.dequantize_e4m3(codes, sc)
    xf = x.double().numpy()
    # the scale is rounded to fp32, so the largest magnitude comes back to within 2^-23
    assert abs(np.abs(back).max() - np.abs(xf).max()) <= 2.0 ** -23 * np.abs(xf).max()
    assert np.float32(sc) == sc
    big = np.abs(xf) > sc * 2.0 ** -6 * 8   # normal range of e4m3
    assert np.all(np.abs(back[big] - xf[big]) <= 2.0 ** -4 * np.abs(xf[big]) + 1e-12)
