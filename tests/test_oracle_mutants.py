"""Planted mistakes in copies of the oracle must be caught by the pins.

Each mutant is the oracle's source with one plausible slip (a dropped term, a
wrong sign, index or operand, a reversed order); it is loaded as a separate
module and every pin check of test_oracle_pins runs against it.  A mutant
that passes all of them would mean the pins cannot see that slip.
"""
import importlib.util
import os

import pytest

import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "dsa_oracle.py")

MUTANTS = {
    "tie_to_higher_position": ("order = np.lexsort((ts, -scores))",
                               "order = np.lexsort((-ts, -scores))"),
    "causal_range_excludes_self": ("return np.arange(prefix_len, pos + 1, dtype=np.int64)",
                                   "return np.arange(prefix_len, pos, dtype=np.int64)"),
    "prefix_scored": ("return np.arange(prefix_len, pos + 1, dtype=np.int64)",
                      "return np.arange(0, pos + 1, dtype=np.int64)"),
    "prefix_dropped": ("return np.concatenate([prefix, np.asarray(idx[:n_sel], dtype=np.int64)])",
                       "return np.asarray(idx[:n_sel], dtype=np.int64)"),
    "scale_dropped": ("z = scale * (q @ kr.T)", "z = (q @ kr.T)"),
    "lse_without_max": ("lse = m[:, 0] + np.log(l)", "lse = np.log(l)"),
    "row_off_by_one": ("rows = positions % BLOCK", "rows = (positions + 1) % BLOCK"),
    "descending_output": ("chosen = np.sort(chosen)", "chosen = np.sort(chosen)[::-1]"),
    "kv_head_ignored": ("return cache[blocks, rows, head]", "return cache[blocks, rows, 0]"),
    "gqa_interleaved_heads": (
        "o, s = softmax_attention(q_heads[g * group:(g + 1) * group], kr, vr, scale)",
        "o, s = softmax_attention(q_heads[g::num_kv_heads], kr, vr, scale)"),
    "score_sign": ("return ts, keys @ np.asarray(q_idx, dtype=np.int64)",
                   "return ts, -(keys @ np.asarray(q_idx, dtype=np.int64))"),
    "k_minus_one": ("chosen = ts[order[:k]]", "chosen = ts[order[:k - 1]]"),
    "slot_block_row_swapped": ("blk, row = divmod(int(slot), BLOCK)",
                               "row, blk = divmod(int(slot), BLOCK)"),
    "window_one_longer": ("return np.arange(max(0, pos - window + 1), pos + 1, dtype=np.int64)",
                          "return np.arange(max(0, pos - window), pos + 1, dtype=np.int64)"),
    "window_excludes_self": ("return np.arange(max(0, pos - window + 1), pos + 1, dtype=np.int64)",
                             "return np.arange(max(0, pos - window + 1), pos, dtype=np.int64)"),
    "heads_share_head0_keys": ("ts, s = index_scores(w[\"q_idx\"][b][g], w[\"idx_cache\"][:, g], bt_row, P, pos)",
                               "ts, s = index_scores(w[\"q_idx\"][b][g], w[\"idx_cache\"][:, 0], bt_row, P, pos)"),
    "heads_attend_head0_rows": ("kr = fetch_rows(w[\"k_cache\"], bt_row, positions, head=g)",
                                "kr = fetch_rows(w[\"k_cache\"], bt_row, positions, head=0)"),
    "value_rows_from_key_cache": ("vr = fetch_rows(v_cache, bt_row, positions, head=g)",
                                  "vr = fetch_rows(k_cache, bt_row, positions, head=g)"),
    "heads_read_head0_table": ("bt_row = w[\"block_table\"][b] if tables is None else tables[g][b]",
                               "bt_row = w[\"block_table\"][b] if tables is None else tables[0][b]"),
    "heads_write_every_head": ("            kc[blk, row, h] = k_new[j, h]\n",
                               "            kc[blk, row] = k_new[j, h]\n"),
}

CHECKS = [getattr(pins, n) for n in dir(pins) if n.startswith("check_")]


def _load_mutant(name, old, new):
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not unique/found"
    spec = importlib.util.spec_from_loader(f"oracle_mutant_{name}", loader=None)
    mod = importlib.util.module_from_spec(spec)
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    mod = _load_mutant(name, *MUTANTS[name])
    caught = []
    for chk in CHECKS:
        try:
            ok = chk(mod)
        except Exception:  # a crash also exposes the mutant
            ok = False
        if not ok:
            caught.append(chk.__name__)
    assert caught, f"mutant {name} passed every pin"
