"""Planted mistakes: the oracle's pins must each catch a plausible error.

Every case copies one oracle function, changes its source text in one or two
places (a dropped term, a wrong sign, index, operand order or rounding rule,
an off-by-one), plants the copy in the oracle in place of the original, and
runs the pins expected to notice; at least one must fail, with an assertion
or with one of the oracle's own argument checks (ValueError).
This checks that the pins tie the oracle to the pages and to the mathematics,
not merely to itself.  CPU only; nothing here touches the CUDA path.
"""
import inspect
import textwrap

import pytest

import oracle
from oracle import formats, layout, method

import test_oracle_formats as TF
import test_oracle_layout as TL
import test_oracle_method as TM


def _mutant(fn, *edits):
    """A copy of fn whose source has each (old, new) replacement applied once."""
    src = textwrap.dedent(inspect.getsource(fn))
    for old, new in edits:
        assert src.count(old) == 1, f"{fn.__name__}: {old!r} does not occur exactly once"
        src = src.replace(old, new)
    ns = dict(fn.__globals__)
    exec(compile(src, f"<mutant of {fn.__module__}.{fn.__name__}>", "exec"), ns)
    return ns[fn.__name__]


def _plant(monkeypatch, fn, mutant):
    """Replace fn by mutant wherever the oracle's modules bind it by name."""
    planted = 0
    for mod in (oracle, method, layout, formats):
        if getattr(mod, fn.__name__, None) is fn:
            monkeypatch.setattr(mod, fn.__name__, mutant)
            planted += 1
    assert planted


# (id, function, edits, pins expected to catch it)
CASES = [
    # group quantizer (the pages' FP8 scale and offset per channel group)
    ("scale-over-2^b", method.quantize,
     [("s = e4m3_round((hi - lo) / qmax)", "s = e4m3_round((hi - lo) / (qmax + 1))")],
     [lambda: TM.test_quantizer_codes_are_exact_nearest_grid_points(4)]),
    ("offset-not-fp8", method.quantize, [("o = e4m3_round(lo)", "o = lo")],
     [lambda: TM.test_quantizer_codes_are_exact_nearest_grid_points(4)]),
    ("clamp-off-by-one", method._nearest_grid_codes, [("k = np.clip(k, 0, qmax)", "k = np.clip(k, 0, qmax - 1)")],
     [lambda: TM.test_quantizer_codes_are_exact_nearest_grid_points(2), TM.test_quantizer_error_bound]),
    ("ties-to-odd", method._nearest_grid_codes,
     [("tie & (np.mod(k, 2.0) != 0.0)", "tie & (np.mod(k, 2.0) == 0.0)")],
     [lambda: TM.test_quantizer_codes_are_exact_nearest_grid_points(4)]),
    ("dequantize-sign", method.dequantize, [("(s * cg + o)", "(s * cg - o)")],
     [TM.test_quantizer_constant_group, TM.test_quantizer_error_bound]),
    # least-squares coefficient and the residual
    ("ls-denominator", method.ls_coefficient, [("den = np.sum(y * y, axis=-1)", "den = np.sum(x * x, axis=-1)")],
     [TM.test_ls_coefficient_minimises_squared_error]),
    ("c-not-bf16", method.compress_group, [("cb = bf16_decode(c_bits)[..., None]", "cb = c[..., None]")],
     [TM.test_residual_uses_bf16_coefficient_and_dequantized_anchor]),
    ("c-against-raw-anchor", method.compress_group,
     [("ref = enc_ref if chained else a_hat", "ref = enc_ref if chained else x[P - 1]")],
     [TM.test_residual_uses_bf16_coefficient_and_dequantized_anchor]),
    ("residual-sign", method.compress_group, [("e = x[j] - cb * ref", "e = x[j] + cb * ref")],
     [lambda: TM.test_reconstruction_error_is_the_residual_quantization_error(False)]),
    ("rotation-transposed", method.compress_group, [("u = e @ R.T", "u = e @ R")],
     [lambda: TM.test_reconstruction_error_is_the_residual_quantization_error(False)]),
    ("rebuild-with-R-not-RT", method.compress_group,
     [("recon[j] = cb * dec_ref + r_hat @ R", "recon[j] = cb * dec_ref + r_hat @ R.T")],
     [lambda: TM.test_reconstruction_error_is_the_residual_quantization_error(False)]),
    ("rebuild-drops-c", method.compress_group,
     [("recon[j] = cb * dec_ref + r_hat @ R", "recon[j] = dec_ref + r_hat @ R")],
     [lambda: TM.test_reconstruction_error_is_the_residual_quantization_error(False)]),
    ("chained-decoder-uses-anchor", method.compress_group,
     [("dec_ref = recon[j + 1] if chained else a_hat", "dec_ref = a_hat")],
     [lambda: TM.test_reconstruction_error_is_the_residual_quantization_error(True)]),
    ("f32-residual-sign", method.compress_group,
     [("e = fma_f32(-cb, ref, x[j])", "e = fma_f32(cb, ref, x[j])")],
     [lambda: TM.test_f32_and_f64_readings_agree_up_to_rounding(False)]),
    ("chained-encoder-drops-c", method.compress_group,
     [("enc_ref = fma_f32(cb, enc_ref, back).astype(np.float64)", "enc_ref = back.astype(np.float64)")],
     [lambda: TM.test_f32_and_f64_readings_agree_up_to_rounding(True)]),
    ("norm-ratio-in-least-squares-mode", method.compress_group,
     [('c = ls_coefficient(x[j], ref) if scaling == "ls" else norm_ratio_coefficient(x[j], ref)',
       'c = norm_ratio_coefficient(x[j], ref) if scaling == "ls" else ls_coefficient(x[j], ref)')],
     [TM.test_residual_uses_bf16_coefficient_and_dequantized_anchor]),
    ("f32-rotate-back-transposed", method.rotate_back_f32,
     [("acc = fma_f32(R[k, :], r[..., k:k + 1], acc)", "acc = fma_f32(R[:, k], r[..., k:k + 1], acc)")],
     [TM.test_f32_rotation_special_cases_and_error_bound]),
    ("f32-rotation-transposed", method.rotate_f32,
     [("u = fma_f32(R[:, k], e[..., k:k + 1], u)", "u = fma_f32(R[k, :], e[..., k:k + 1], u)")],
     [TM.test_f32_rotation_special_cases_and_error_bound]),
    ("norm-ratio-without-sqrt", method.norm_ratio_coefficient,
     [("np.sqrt(num / np.where(den > 0, den, 1.0))", "num / np.where(den > 0, den, 1.0)")],
     [TM.test_norm_ratio_coefficient]),
    # Walsh-Hadamard rotation
    ("butterfly-sign", method.fwht_f32, [("np.stack([a + b, a - b]", "np.stack([a + b, b - a]")],
     [lambda: TM.test_fwht_is_the_sylvester_matrix_exactly(8)]),
    ("hadamard-normalisation", method.hadamard_f32, [("np.float32(1.0 / np.sqrt(d))", "np.float32(1.0 / d)")],
     [TM.test_hadamard_rotation_close_to_the_dense_product]),
    # attention
    ("attention-drops-scale", method.attention, [("s = scale * (K @ q)", "s = K @ q")],
     [TM.test_attention_special_cases]),
    ("attention-mean-not-softmax-sum", method.attention, [("return (p @ V) / np.sum(p)", "return (p @ V) / len(p)")],
     [TM.test_attention_special_cases]),
    ("current-token-K-from-V", oracle.decode_attention,
     [("K = np.concatenate([K, k_cur[b, h][None, :]], axis=0)", "K = np.concatenate([K, v_cur[b, h][None, :]], axis=0)")],
     [TL.test_decode_attention_over_cache]),
    ("gqa-head-modulo", oracle.decode_attention, [("h = qh // qpk", "h = qh % H")],
     [TL.test_grouped_query_attention_is_multi_head_over_copied_kv_heads]),
    # rebuild from the cache bytes, and the current token's append
    ("reader-rebuilds-with-R", oracle.reconstruct,
     [("x = bf16_decode(cbits)[:, None] * x + r_hat @ R", "x = bf16_decode(cbits)[:, None] * x + r_hat @ R.T")],
     [lambda: TL.test_decode_attention_append_writes_the_next_slot(False)]),
    ("reader-chained-reads-one-plane", oracle.reconstruct,
     [("js = range(P - 2, loop - 1, -1) if chained else [loop]", "js = [loop]")],
     [lambda: TL.test_decode_attention_append_writes_the_next_slot(True)]),
    ("append-slot-off-by-one", oracle.decode_attention_append,
     [("np.where(ok, seq, 0)", "np.where(ok, seq + 1, 0)")],
     [lambda: TL.test_decode_attention_append_writes_the_next_slot(False)]),
    ("append-capacity-off-by-one", oracle.decode_attention_append,
     [("ok = (seq >= 0) & (seq + 1 <= geom.max_seq_len)", "ok = (seq >= 0) & (seq + 2 <= geom.max_seq_len)")],
     [lambda: TL.test_decode_attention_append_writes_the_next_slot(False)]),
    # byte layout and storage accounting
    ("nibble-order", layout._code_addresses,
     [("shift = (ch[None, :] % per_byte) * bits", "shift = (per_byte - 1 - ch[None, :] % per_byte) * bits")],
     [TL.test_code_positions_in_bytes]),
    ("v-word-token-order", layout._code_addresses,
     [("byte_in_row = 4 * word + (q % 4)", "byte_in_row = 4 * word + q // per_byte"),
      ("slot = q // 4", "slot = q % per_byte")],
     [lambda: TL.test_channel_major_masks_give_consecutive_tokens(4)]),
    ("writer-swaps-scale-and-offset", layout.pack_group,
     [("buf[ma] = a_s[kv, b, h]\n                buf[ma + 1] = a_o[kv, b, h]",
       "buf[ma] = a_o[kv, b, h]\n                buf[ma + 1] = a_s[kv, b, h]")],
     [lambda: TL.test_decode_attention_append_writes_the_next_slot(False)]),
    ("writer-c-big-endian", layout.pack_group,
     [("buf[ca] = (cb & 0xFF).astype(np.uint8)\n                    buf[ca + 1] = (cb >> 8).astype(np.uint8)",
       "buf[ca] = (cb >> 8).astype(np.uint8)\n                    buf[ca + 1] = (cb & 0xFF).astype(np.uint8)")],
     [lambda: TL.test_decode_attention_append_writes_the_next_slot(False)]),
    ("storage-drops-coefficient", layout.bits_per_element,
     [("resid = 8.0 * (head_dim / 4 + 2 * ng + 2) / head_dim", "resid = 8.0 * (head_dim / 4 + 2 * ng) / head_dim")],
     [TL.test_storage_accounting_reproduces_the_pages]),
    ("paged-head-order", layout.paged_pool,
     [("dst = ((layer * G + group) * num_pages + page) * page_bytes + h * head_block",
       "dst = ((layer * G + group) * num_pages + page) * page_bytes + (H - 1 - h) * head_block")],
     [TL.test_paged_pool_moves_whole_tiles]),
    # number formats
    ("rounding-ties-up", formats._round_to_format,
     [("k = np.rint(ax / quantum)", "k = np.floor(ax / quantum + 0.5)")],
     [TF.test_e4m3_midpoints_brute_force, TF.test_bf16_matches_torch_cast_from_fp32]),
    ("e4m3-no-saturation", formats.e4m3_round,
     [("np.clip(x, -E4M3_MAX, E4M3_MAX), _E4M3_MANT_BITS", "x, _E4M3_MANT_BITS"),
      ("return np.clip(r, -E4M3_MAX, E4M3_MAX)", "return r")],
     [lambda: TF.test_e4m3_fixed_points(500.0, 0x7E)]),
    ("e4m3-negative-zero-loses-sign", formats.e4m3_encode, [("neg = np.signbit(x)", "neg = x < 0")],
     [TF.test_e4m3_negative_underflow_keeps_sign]),
    ("e4m3-encode-bias", formats.e4m3_encode,
     [("norm_e = np.clip(e_unb + 7, 1, 15)", "norm_e = np.clip(e_unb + 8, 1, 15)")],
     [TF.test_e4m3_encode_matches_torch_cast_in_range]),
    ("e4m3-decode-bias", formats.e4m3_decode,
     [("np.ldexp(1.0, (e - 7).astype(np.int32))", "np.ldexp(1.0, (e - 8).astype(np.int32))")],
     [TF.test_e4m3_decode_matches_torch_on_all_bytes]),
    ("fma-rounds-twice", formats.fma_f32,
     [("return _round_to_odd_sum(p, np.broadcast_to(c, p.shape).astype(np.float64)).astype(np.float32)",
       "return (p + np.broadcast_to(c, p.shape)).astype(np.float32)")],
     [TM.test_fma_f32_is_one_rounding_of_the_exact_value]),
]


@pytest.mark.parametrize("name,fn,edits,pins", CASES, ids=[c[0] for c in CASES])
def test_a_planted_mistake_fails_a_pin(name, fn, edits, pins, monkeypatch):
    _plant(monkeypatch, fn, _mutant(fn, *edits))
    caught = 0
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError):
            caught += 1
    assert caught, f"no pin noticed the planted mistake {name!r}"


def test_the_unmutated_copies_pass_the_same_pins(monkeypatch):
    """The copying itself changes nothing: every function recompiled from its
    unedited source passes the pins of its cases."""
    seen = set()
    for name, fn, _, pins in CASES:
        if fn in seen:
            continue
        seen.add(fn)
        _plant(monkeypatch, fn, _mutant(fn))
    for name, fn, _, pins in CASES[:8]:
        for pin in pins:
            pin()
