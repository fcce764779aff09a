"""Plant plausible mistakes in copies of the oracle (on the CPU) and show that
the pins catch every one of them.

Each mutant is the oracle's own module source with one edit -- a dropped term,
a flipped sign, a wrong index or a transposed operand -- executed into a fresh
namespace.  The pin checks of oracle_pins.py must fail for at least one check
per mutant; otherwise the pins would not be strong enough to trust the
oracle.
"""

import inspect
import types

import pytest

import oracle.attention as attention
import oracle_pins

MUTANTS = {
    "scores_drop_scale": ("    s = scale * (q @ k.T)\n    if causal:\n        i = np.arange(s.shape[0])",
                          "    s = (q @ k.T)\n    if causal:\n        i = np.arange(s.shape[0])"),
    "cached_scores_drop_scale": ("    s = scale * (q @ k.T)\n    if causal:\n        nq, nk = s.shape",
                                 "    s = (q @ k.T)\n    if causal:\n        nq, nk = s.shape"),
    "mask_strict_lower": ("        s = np.where(j <= i, s, -np.inf)\n    return s",
                          "        s = np.where(j < i, s, -np.inf)\n    return s"),
    "mask_upper": ("        s = np.where(j <= i, s, -np.inf)\n    return s",
                   "        s = np.where(j >= i, s, -np.inf)\n    return s"),
    "softmax_wrong_axis": ("    l = e.sum(axis=1)\n    L = np.where",
                           "    l = e.sum(axis=0)\n    L = np.where"),
    "lse_missing_log": ("m0 + np.log(np.where(has_key, l, 1.0))",
                        "m0 + np.where(has_key, l, 1.0)"),
    "lse_missing_max": ("m0 + np.log(np.where(has_key, l, 1.0))",
                        "np.log(np.where(has_key, l, 1.0))"),
    "output_transposed_weights": ("    O = P @ _f64(v)\n    return O, L",
                                  "    O = P.T @ _f64(v)\n    return O, L"),
    "online_rescale_sign": ("rescale = np.exp(m - m_new) if np.isfinite(m) else 0.0",
                            "rescale = np.exp(m_new - m) if np.isfinite(m) else 0.0"),
    "online_l_not_rescaled": ("        l = rescale * l + e.sum()\n",
                              "        l = l + e.sum()\n"),
    "online_u_not_rescaled": ("        u = rescale * u + e @ values[a:b]\n",
                              "        u = u + e @ values[a:b]\n"),
    "dS_sign": ("    dS = P * (dP - D[:, None])\n    dQ = scale * (dS @ k)",
                "    dS = P * (dP + D[:, None])\n    dQ = scale * (dS @ k)"),
    "dK_missing_transpose": ("    dK = scale * (dS.T @ q)\n    return dQ, dK, dV, D",
                             "    dK = scale * (dS @ q)\n    return dQ, dK, dV, D"),
    "dK_wrong_operand": ("    dK = scale * (dS.T @ q)\n    return dQ, dK, dV, D",
                         "    dK = scale * (dS.T @ k)\n    return dQ, dK, dV, D"),
    "dQ_missing_scale": ("    dQ = scale * (dS @ k)\n    dK",
                         "    dQ = (dS @ k)\n    dK"),
    "D_missing_P": ("    D = (P * dP).sum(axis=1) if o_stored is None else (do * _f64(o_stored)).sum(axis=1)\n"
                    "    dS = P * (dP - D[:, None])\n    dQ = scale",
                    "    D = dP.sum(axis=1) if o_stored is None else (do * _f64(o_stored)).sum(axis=1)\n"
                    "    dS = P * (dP - D[:, None])\n    dQ = scale"),
    "stored_o_ignored": ("    D = (P * dP).sum(axis=1) if o_stored is None else (do * _f64(o_stored)).sum(axis=1)\n"
                         "    dS = P * (dP - D[:, None])\n    dQ = scale",
                         "    D = (P * dP).sum(axis=1)\n    dS = P * (dP - D[:, None])\n    dQ = scale"),
    "stored_o_wrong_operand": ("    D = (P * dP).sum(axis=1) if o_stored is None else (do * _f64(o_stored)).sum(axis=1)\n"
                               "    dS = P * (dP - D[:, None])\n    dQ = scale",
                               "    D = (P * dP).sum(axis=1) if o_stored is None else (v * _f64(o_stored)).sum(axis=1)\n"
                               "    dS = P * (dP - D[:, None])\n    dQ = scale"),
    "stored_o_wrong_head": ("                q[b, h], k[b, h], v[b, h], do[b, h], scale, causal,\n"
                            "                None if o_stored is None else o_stored[b, h])",
                            "                q[b, h], k[b, h], v[b, h], do[b, h], scale, causal,\n"
                            "                None if o_stored is None else o_stored[h % B, b % H])"),
    "dropout_D_missing_P": ("    D = (P * dP).sum(axis=1) if o_stored is None else (do * _f64(o_stored)).sum(axis=1)\n"
                            "    dS = P * (dP - D[:, None])\n    return scale",
                            "    D = dP.sum(axis=1) if o_stored is None else (do * _f64(o_stored)).sum(axis=1)\n"
                            "    dS = P * (dP - D[:, None])\n    return scale"),
    "dropout_stored_o_ignored": ("    D = (P * dP).sum(axis=1) if o_stored is None else (do * _f64(o_stored)).sum(axis=1)\n"
                                 "    dS = P * (dP - D[:, None])\n    return scale",
                                 "    D = (P * dP).sum(axis=1)\n    dS = P * (dP - D[:, None])\n    return scale"),
    "dV_missing_transpose": ("    dV = P.T @ do\n    dP = do @ v.T",
                             "    dV = P @ do\n    dP = do @ v.T"),
    "cached_mask_top_left": ("        s = np.where(j <= i + (nk - nq), s, -np.inf)",
                             "        s = np.where(j <= i, s, -np.inf)"),
    "cached_mask_off_by_one": ("        s = np.where(j <= i + (nk - nq), s, -np.inf)",
                               "        s = np.where(j < i + (nk - nq), s, -np.inf)"),
    "cached_mask_sign": ("        s = np.where(j <= i + (nk - nq), s, -np.inf)",
                         "        s = np.where(j <= i - (nk - nq), s, -np.inf)"),
    "cached_output_values_swapped": ("    return P @ _f64(v), L\n",
                                     "    return P @ _f64(k), L\n"),
    "philox_words_swapped": ("        c = [(p1 >> np.uint64(32)) ^ c[1] ^ np.uint64(k0), p1 & mask,",
                             "        c = [(p1 >> np.uint64(32)) ^ c[3] ^ np.uint64(k0), p1 & mask,"),
    "philox_key_not_advanced": ("        k1 = (k1 + _PHILOX_W1) & 0xFFFFFFFF\n",
                                "        k1 = k1\n"),
    "dropout_keep_inverted": ("    return w.astype(np.float64) / 2.0**32 >= p\n",
                              "    return w.astype(np.float64) / 2.0**32 < p\n"),
    "dropout_no_rescale": ("    return (P * keep / (1.0 - p)) @ _f64(v), L\n",
                           "    return (P * keep) @ _f64(v), L\n"),
    "dropout_dP_unmasked": ("    dP = (do @ v.T) * M\n", "    dP = (do @ v.T)\n"),
    "dropout_dV_unmasked": ("    dV = (P * M).T @ do\n", "    dV = P.T @ do\n"),
    "dP_transposed": ("    dV = P.T @ do\n    dP = do @ v.T",
                      "    dV = P.T @ do\n    dP = v @ do.T"),
}


def _mutant_module(old, new):
    src = inspect.getsource(attention)
    assert src.count(old) == 1, f"mutation site not unique: {old!r}"
    ns = {"__name__": "oracle_mutant"}
    exec(compile(src.replace(old, new), "<oracle-mutant>", "exec"), ns)
    return types.SimpleNamespace(**{k: v for k, v in ns.items() if not k.startswith("__")})


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    impl = _mutant_module(*MUTANTS[name])
    caught = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(impl)
        except Exception:   # an assertion, or a shape error the mistake causes
            caught.append(check.__name__)
    assert caught, f"no pin detects mutant {name}"


def test_unmutated_copy_passes():
    src = inspect.getsource(attention)
    ns = {"__name__": "oracle_copy"}
    exec(compile(src, "<oracle-copy>", "exec"), ns)
    impl = types.SimpleNamespace(**{k: v for k, v in ns.items() if not k.startswith("__")})
    for check in oracle_pins.ALL_CHECKS:
        check(impl)
