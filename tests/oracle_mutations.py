"""Planted mistakes in the oracle (test infrastructure, CPU only).

Each entry changes one expression of one oracle module -- a plausible slip:
a dropped or swapped term, a wrong sign, constant or index, an operand on the
wrong side -- and names the pin files that must then fail.  ``plant(name)``
executes the changed source in the live module, so every importer of the
module sees the mistake.  ``tests/test_oracle_mutations.py`` runs the pins
once per entry in a child process with ``QMUON_PLANT_ORACLE_MISTAKE`` set
(``conftest.py`` plants it) and requires a failure each time.

Changes that leave the mathematics intact are not listed: skipping ColNorm
before the thin QR, for one, scales the columns of M_t Q by positive numbers
and so gives the same positive-diagonal factor P; nor does restoring the
blocks outside every group after the in-place normalisation, whose scale
there is already 1.
"""

import importlib
import inspect

CODEC = ["test_oracle_codec.py"]
NS = ["test_oracle_ns.py"]
CARRIER = ["test_oracle_carrier.py"]
SR = ["test_oracle_sr.py"]
GRASP = ["test_oracle_grasp.py"]

# name: (module, expression, replacement, pin files)
MUTATIONS = {
    # codec ("Quantized Muon Momentum", section "Algorithm")
    "ema_gradient_weight_beta": ("oracle.codec", "(omb * g).astype(F32)", "(beta32 * g).astype(F32)", CODEC),
    "ema_state_weight_one_minus_beta": ("oracle.codec", "(beta32 * old)", "(omb * old)", CODEC),
    "dequant_scale_over_128": ("oracle.codec", "s_old = (absmax / F32(127.0))", "s_old = (absmax / F32(128.0))", CODEC),
    "requant_ties_away_from_zero": ("oracle.codec", "r = np.rint(x)", "r = np.trunc(x + np.copysign(0.5, x))", CODEC),
    "requant_truncates": ("oracle.codec", "r = np.rint(x)", "r = np.trunc(x)", CODEC),
    "uint8_offset_127": ("oracle.codec", "astype(np.int32) - 128", "astype(np.int32) - 127", CODEC),
    "bf16_truncates": ("oracle.codec", "((u + 0x7FFF + lsb) >> 16)", "(u >> 16)", CODEC),
    "absmax_of_signed_values": ("oracle.codec", "np.fmax.reduce(np.abs(m), axis=1", "np.fmax.reduce(m, axis=1", CODEC),
    "group_sum_of_abs_not_squares": ("oracle.codec", "block_sumsq = np.sum(m64 * m64, axis=1)",
                                     "block_sumsq = np.sum(np.abs(m64), axis=1)", CODEC),
    "inverse_norm_eps_inside_sqrt": ("oracle.codec", "(1.0 / (np.sqrt(S) + EPS))", "(1.0 / np.sqrt(S + EPS))",
                                     CODEC),
    "bf16_ties_away": ("oracle.codec", "lsb = (u >> 16) & 1", "lsb = 1", CODEC),
    "one_minus_beta_in_fp64": ("oracle.codec", "omb = F32(F32(1.0) - beta32)", "omb = F32(1.0 - float(beta))", CODEC),
    "tail_padding_kept": ("oracle.codec", "m.reshape(-1)[numel:] = 0.0", "m.reshape(-1)[numel:] = 1.0", CODEC),
    "zero_block_codes_not_forced": ("oracle.codec", "qn = np.where(amax[:, None] == 0, 0, qn)",
                                    "qn = np.where(amax[:, None] == 0, 1, qn)", CODEC),
    "segment_overlap_allowed": ("oracle.codec", "if np.any(arr[b0:b1] >= 0):", "if False:", CODEC),
    "absmax_propagates_nan": ("oracle.codec", "amax = np.fmax.reduce(np.abs(m), axis=1", "amax = np.maximum.reduce(np.abs(m), axis=1",
                              CODEC),
    "nan_code_not_zeroed": ("oracle.codec", "r = np.where(np.isnan(r), 0.0, r)", "r = np.where(np.isnan(r), 127.0, r)",
                            CODEC),
    "group_sum_overwrites": ("oracle.codec", "S[g] += float(np.sum(bs[sel]))", "S[g] = float(np.sum(bs[sel]))", CODEC),
    "segment_drops_partial_last_block": ("oracle.codec", "b0, b1 = s.start // QBLOCK, n_blocks(end)",
                                         "b0, b1 = s.start // QBLOCK, end // QBLOCK", CODEC),
    "eps_1e6": ("oracle.codec", "EPS = 1e-7", "EPS = 1e-6", CODEC),
    "fp16_store_truncates": ("oracle.codec", "return np.asarray(m, dtype=F32).astype(np.float16)  # IEEE nearest-even",
                             "return np.trunc(np.asarray(m, dtype=F32) * 1024).astype(np.float16) / 1024", CODEC),
    "normalize_divides": ("oracle.codec", "scaled = (g32 * scale[:, None])", "scaled = (g32 / scale[:, None])", CODEC),
    "segment_tail_rejected": ("oracle.codec", "(end % QBLOCK and end != n)", "(end % QBLOCK)", CODEC),
    "dequantize_over_128": ("oracle.codec", "(np.asarray(absmax, dtype=F32) / F32(127.0))",
                            "(np.asarray(absmax, dtype=F32) / F32(128.0))", CODEC),
    # Newton-Schulz ("NVIDIA impulsa ... Megatron", section "Newton-Schulz distribuido")
    "ns_poly_sign_of_c": ("oracle.ns", "B = b * A + c * (A @ A)", "B = b * A - c * (A @ A)", NS),
    "ns_drops_a_term": ("oracle.ns", "X = a * X + B @ X", "X = B @ X", NS),
    "ns_update_on_the_right": ("oracle.ns", "X = a * X + B @ X", "X = a * X + X @ B", NS),
    "ns_gram_transposed": ("oracle.ns", "A = X @ X.T", "A = X.T @ X", NS),
    "ns_coefficients_reversed": ("oracle.ns", "a, b, c = (float(v) for v in coeffs)",
                                 "c, b, a = (float(v) for v in coeffs)", NS),
    "ns_inverse_norm_divides": ("oracle.ns", "X = X * float(inv_norm)", "X = X / float(inv_norm)", NS),
    # MuonBP ("MuonBP: Faster Muon via Block-Periodic Orthogonalization", section "整体框架")
    "muonbp_full_step_offset": ("oracle.muonbp", "return P != 0 and t % P == 0", "return P != 0 and t % P == 1", NS),
    "muonbp_learning_rates_swapped": ("oracle.muonbp", "eta = F32(eta_full if full else eta_block)",
                                      "eta = F32(eta_block if full else eta_full)", NS),
    "muonbp_shared_tile_norm": ("oracle.muonbp", "inv_norm=float(inv[g])", "inv_norm=float(inv[gbase])", NS),
    "muonbp_row_tile_offset": ("oracle.muonbp", "segs.append(codec.NormSegment(tensor_index, i * th * cols, th * cols, g))",
                               "segs.append(codec.NormSegment(tensor_index, i * th, th * cols, g))", NS),
    "muonbp_group_base_step": ("oracle.muonbp", "gbase += tr * tc", "gbase += 1", NS),
    "muonbp_weight_step_sign": ("oracle.muonbp", "W = (s.weight.astype(F32) - (eta * u32).astype(F32)).astype(F32)",
                                "W = (s.weight.astype(F32) + (eta * u32).astype(F32)).astype(F32)", NS),
    "muonbp_update_applied_unrounded": ("oracle.muonbp", "u32 = codec.f32_from_bf16_bits(ub).reshape(s.rows, s.cols)",
                                        "u32 = U.astype(F32)", NS),
    "muonbp_tile_column_offset": ("oracle.muonbp", "r * cols + j * tw", "r * cols + j * th", NS),
    # MXFP8 carrier ("Quantized Muon Momentum", section "Wave18B MXFP8 Carrier Probe")
    "e4m3_subnormal_exponent": ("oracle.carrier", "2.0 ** (1 - 7)", "2.0 ** (0 - 7)", CARRIER),
    "e4m3_ties_to_odd": ("oracle.carrier", "(lo % 2 == 0)", "(lo % 2 == 1)", CARRIER),
    "e4m3_bias_8": ("oracle.carrier", "2.0 ** (e - 7)", "2.0 ** (e - 8)", CARRIER),
    "e8m0_not_minimal": ("oracle.carrier", "while amax > math.ldexp(E4M3_MAX, e)",
                         "while amax >= math.ldexp(E4M3_MAX, e)", CARRIER),
    "e8m0_zero_block_byte": ("oracle.carrier", "return 127 if amax == 0.0 else 254", "return 0 if amax == 0.0 else 254",
                             CARRIER),
    "carrier_decode_scale_stride": ("oracle.carrier", "np.repeat(e8m0_value(scale_inv), SCALE_BLOCK, axis=1)",
                                    "np.tile(e8m0_value(scale_inv), (1, SCALE_BLOCK))", CARRIER),
    "carrier_scale_inverted": ("oracle.carrier", "127 - bytes_.astype(np.int64)", "bytes_.astype(np.int64) - 127",
                               CARRIER),
    "carrier_norm_without_root": ("oracle.carrier", "(math.sqrt(S) + codec.EPS)", "(S + codec.EPS)", CARRIER),
    # Philox4x32-10 (Salmon et al., SC'11) for the stochastic requantisation
    "philox_multiplier": ("oracle.rng", "M0 = 0xD2511F53\n", "M0 = 0xD2511F55\n", SR),
    "philox_key_bumped_before_round_one": ("oracle.rng", "if r > 0:", "if r >= 0:", SR),
    "philox_words_crossed": ("oracle.rng", "(p1 >> np.uint64(32)) ^ c1 ^ k0", "(p0 >> np.uint64(32)) ^ c1 ^ k0", SR),
    "sr_floor_replaced_by_rint": ("oracle.codec", "r = np.floor(x.astype(np.float64) + u)",
                                  "r = np.rint(x.astype(np.float64) + u - 0.5)", SR),
    "sr_counter_tensor_word_is_step": ("oracle.rng", "ctr[:, 2] = np.uint64(tensor_index & _MASK)",
                                       "ctr[:, 2] = np.uint64(step & _MASK)", SR),
    "sr_uniform_scale_2_23": ("oracle.rng", "* 2.0 ** -24", "* 2.0 ** -23", SR),
    # GRASP ("4-bit-Muon-GRASP", the update equations and the grid quantisation)
    "grasp_grid_uses_max": ("oracle.grasp", "return np.minimum(rb, cb).astype(F32)",
                            "return np.maximum(rb, cb).astype(F32)", GRASP),
    "grasp_reconstruct_subtracts": ("oracle.grasp", "return (res + acc).astype(F32)",
                                    "return (res - acc).astype(F32)", GRASP),
    "grasp_residual_sign": ("oracle.grasp", "resid = mt - p @ r.T", "resid = mt + p @ r.T", GRASP),
    "grasp_levels_2_pow_b_minus_1": ("oracle.grasp", "L = F32(2 ** (bits - 1) - 1)\n    nbr",
                                     "L = F32(2 ** (bits - 1))\n    nbr", GRASP),
    "grasp_dequant_step_times_level": ("oracle.grasp", "step = (d / L).astype(F32)", "step = (d * L).astype(F32)",
                                       GRASP),
    "grasp_row_max_over_whole_row": ("oracle.grasp", "rmax[bj] = a[:, bj * s_cols:(bj + 1) * s_cols].max(axis=1)",
                                     "rmax[bj] = a.max(axis=1)", GRASP),
    "grasp_qr_sign_not_fixed": ("oracle.grasp", "sgn = np.where(np.diag(rf) < 0, -1.0, 1.0)",
                                "sgn = np.ones(rf.shape[0])", GRASP),
    "grasp_column_max_over_whole_column": ("oracle.grasp", "cmax[bi] = a[bi * s_rows:(bi + 1) * s_rows, :].max(axis=0)",
                                           "cmax[bi] = a.max(axis=0)", GRASP),
    "grasp_grid_truncates": ("oracle.grasp", "q = np.rint((x * sc).astype(F32))", "q = np.trunc((x * sc).astype(F32))",
                             GRASP),
    "grasp_nibbles_swapped": ("oracle.grasp", "(u[:, 0::2] | (u[:, 1::2] << 4))", "(u[:, 1::2] | (u[:, 0::2] << 4))",
                              GRASP),
    "grasp_momentum_mu_on_gradient": ("oracle.grasp", "m = ((F32(mu) * m_prev).astype(F32) + g).astype(F32)",
                                      "m = (m_prev + (F32(mu) * g).astype(F32)).astype(F32)", GRASP),
}


def plant(name: str) -> None:
    """Execute the oracle module of ``name`` with its one expression changed."""
    mod_name, old, new, _ = MUTATIONS[name]
    mod = importlib.import_module(mod_name)
    src = inspect.getsource(mod)
    if src.count(old) != 1:
        raise RuntimeError(f"{name}: the expression {old!r} occurs {src.count(old)} times in {mod_name}")
    exec(compile(src.replace(old, new), mod.__file__, "exec"), mod.__dict__)
