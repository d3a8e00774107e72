"""Planted mistakes: every plausible slip in the oracle makes at least one of its pins fail.

Each case below rewrites one line of one oracle function on the CPU (a flipped sign, an
off-by-one window or block bound, a dropped normalisation, a swapped operand, a wrong tie rule, a
missing rounding), installs the rewritten function wherever the original is referenced (the
oracle's own modules and the pin modules), and runs the pins that cover that function:
``tests/test_oracle_*.py``.  The case passes when at least one pin fails under the mistake, which
is what shows the pins tie the oracle to the report's definitions rather than to itself.  The
real oracle is untouched: the rewrite lives only inside the test (pytest's monkeypatch undoes it).
"""

import inspect
import sys
import textwrap

import pytest

import oracle.accept
import oracle.compress
import oracle.indexer
import oracle.plan
import oracle.refresh
import oracle.round
import oracle.storage
import oracle.verify
import test_oracle_accept as p_accept
import test_oracle_compress as p_compress
import test_oracle_indexer as p_indexer
import test_oracle_plan as p_plan
import test_oracle_refresh as p_refresh
import test_oracle_storage as p_storage
import test_oracle_verify as p_verify


def _mutant(func, old, new):
    """``func`` with the single occurrence of ``old`` in its source replaced by ``new``."""
    src = textwrap.dedent(inspect.getsource(func))
    assert src.count(old) == 1, f"{func.__name__}: {old!r} must occur exactly once"
    ns = dict(func.__globals__)
    exec(compile(src.replace(old, new), inspect.getsourcefile(func), "exec"), ns)
    return ns[func.__name__]


def _install(monkeypatch, func, mutant):
    """Replace every module-level reference to ``func`` in the oracle and pin modules."""
    n = 0
    for name, mod in list(sys.modules.items()):
        if not (name == "oracle" or name.startswith("oracle.") or name.startswith("test_oracle_")):
            continue
        for attr, val in list(vars(mod).items()):
            if val is func:
                monkeypatch.setattr(mod, attr, mutant)
                n += 1
    assert n > 0


def _fails(pin):
    try:
        pin()
    except Exception:   # an assertion, or the oracle raising on its own checks
        return True
    return False


# pins by the oracle function they cover (called lazily, with the parameters pytest would use)
def _verify_a():
    return [lambda c=c: p_verify.test_check_a_every_node_equals_linear_decode(c)
            for c in range(len(p_verify.CASES))]


def _verify_all():
    return _verify_a() + [
        lambda: p_verify.test_check_b_chain_equals_sequential_decode_with_commits("f64"),
        lambda: p_verify.test_check_b_chain_equals_sequential_decode_with_commits("bf16"),
        p_verify.test_single_visible_entry_returns_its_value,
        p_verify.test_zero_query_gives_mean_of_visible_values_and_lse_is_logsumexp,
        p_verify.test_selection_list_restricts_persistent_c4_only,
    ]


def _compress():
    return [lambda m=m, d=d: p_compress.test_gated_sum_closed_form(m, d)
            for m, d in [(4, 16), (4, 64), (128, 8), (16, 32)]] + [
        p_compress.test_zero_gate_gives_block_mean,
        p_compress.test_identical_rows_give_that_row,
        p_compress.test_dominant_logit_selects_that_token,
        p_compress.test_permutation_invariance_and_gate_shift,
        lambda: p_compress.test_vectorised_blocks_equal_per_block_definition(4),
        lambda: p_compress.test_vectorised_blocks_equal_per_block_definition(128),
        p_compress.test_many_blocks_span_several_slabs,
    ]


def _plan():
    return [p_plan.test_golden_tiny_tree, p_plan.test_chain_closed_form,
            p_plan.test_star_closed_form, p_plan.test_remainder_tail_bounds] + [
        lambda s=s: p_plan.test_random_tree_against_reachability(s) for s in range(20)]


def _accept():
    return [p_accept.test_golden_tiny, p_accept.test_single_node,
            p_accept.test_all_mismatch_and_all_match_chain,
            p_accept.test_lowest_index_child_wins_a_tie] + [
        lambda s=s: p_accept.test_random_trees_against_enumeration(s) for s in range(30)]


def _refresh():
    return [lambda st=st, L=L, n=n: p_refresh.test_refresh_equals_compress_from_scratch(st, L, n)
            for st in ("bf16", "f64")
            for L, n in [(250, 8), (253, 3), (255, 1), (127, 4), (120, 8)]] + [
        p_refresh.test_capacity_is_enforced, p_refresh.test_commit_fills_every_capacity_exactly,
        p_refresh.test_tiny_round_golden]


def _round():
    return [p_refresh.test_tiny_round_golden] + [
        lambda L=L: p_refresh.test_round_reports_the_rows_and_entries_it_commits(L)
        for L in (250, 253)]


def _indexer():
    return [p_indexer.test_integer_scores_equal_the_exact_dot_product,
            p_indexer.test_scores_round_in_index_order,
            p_indexer.test_topk_special_cases,
            p_indexer.test_select_uses_only_the_complete_blocks] + [
        lambda s=s: p_indexer.test_topk_matches_brute_force_with_ties(s) for s in range(12)]


def _storage():
    return [p_storage.test_bf16_matches_torch_on_fp32_values,
            p_storage.test_bf16_matches_exact_rational_on_fp64_values,
            p_storage.test_f32_matches_exact_rational, p_storage.test_f64_is_identity]


C, P, V, A, R, I, S, RD = (oracle.compress, oracle.plan, oracle.verify, oracle.accept,
                           oracle.refresh, oracle.indexer, oracle.storage, oracle.round)

MUTANTS = [
    # compressor ([TSD-V4] §2.2, the gated-sum stand-in)
    ("gate logit sign flipped", C.gated_block_sum, "z = Kb @ g", "z = -(Kb @ g)", _compress),
    ("gate weights not normalised", C.gated_block_sum, "w = w / w.sum()", "w = w / len(w)",
     _compress),
    ("value entry built from keys", C.gated_block_sum, "return w @ Kb, w @ Vb",
     "return w @ Kb, w @ Kb", _compress),
    ("block read one row late", C.compress_blocks, "t0 = m * (j - s0)", "t0 = m * (j - s0) + 1",
     _compress),
    ("slab start not subtracted", C.compress_blocks, "t0 = m * (j - s0)", "t0 = m * j", _compress),
    # plan ([TSD-V4] §3.1, §4.1)
    ("window one token short", P.build_plan, "max(0, pos[v] - W)", "max(0, pos[v] - W + 1)",
     lambda: _plan() + _verify_a()),
    ("block completion off by one", P.build_plan, "(pos[v] + 1) % m == 0", "pos[v] % m == 0",
     lambda: _plan() + _verify_a()),
    ("node sees its own scratch entry", P.build_plan, "if u != v and (anc[v] >> u) & 1",
     "if (anc[v] >> u) & 1", lambda: _plan() + _verify_a()),
    ("positions start one past L", P.build_plan, "pos = [L + depth[v] for v in range(D)]",
     "pos = [L + depth[v] + 1 for v in range(D)]", lambda: _plan() + _verify_a()),
    ("remainder tail rounds up", P.build_plan, "m_min * (pos[v] // m_min)",
     "m_min * ((pos[v] + 1) // m_min)", lambda: _plan() + _verify_a()),
    ("window not clamped at 0", P.build_plan, "raw_lo = [max(0, pos[v] - W) for v in range(D)]",
     "raw_lo = [pos[v] - W for v in range(D)]", lambda: _plan() + _verify_a()),
    ("scratch visibility tests the viewer", P.build_plan, "(anc[v] >> u) & 1 and completes[m][u]",
     "(anc[v] >> u) & 1 and completes[m][v]", lambda: _plan() + _verify_a()),
    # verify ([TSD-V4] §3.1, §3.2, §4.2)
    ("scratch visibility transposed", V.visible_set, "if (plan.scr_vis[m][v] >> u) & 1:",
     "if (plan.scr_vis[m][u] >> v) & 1:", _verify_all),
    ("scratch block ends one early", V.scratch_entries, "end = plan.pos[u]", "end = plan.pos[u] - 1",
     _verify_all),
    ("logit scale 1/d", V.attend, "/ math.sqrt(d)", "/ d", _verify_all),
    ("LSE in log2", V.attend, "LSE = (M + np.log(Z))[:, 0]", "LSE = (M + np.log2(Z))[:, 0]",
     _verify_all),
    ("values replaced by keys", V.attend, "O = (E @ Vvis) / Z", "O = (E @ Kvis) / Z", _verify_all),
    ("raw tail starts one late", V.visible_set, "for t in range(plan.raw_lo[v], L):",
     "for t in range(plan.raw_lo[v] + 1, L):", _verify_all),
    ("last persistent entry dropped", V.visible_set, "n = L // m", "n = max(0, L // m - 1)",
     _verify_all),
    ("tree token at the window edge hidden", V.visible_set, "plan.pos[u] >= plan.raw_lo[v]",
     "plan.pos[u] > plan.raw_lo[v]", _verify_all),
    ("ancestor tokens ignored", V.visible_set, "if (plan.anc[v] >> u) & 1 and plan.pos[u]",
     "if u == v and plan.pos[u]", _verify_all),
    ("selection applied to C128 too", V.visible_set, "if m == 4 and sel is not None:",
     "if sel is not None:", _verify_all),
    ("scratch block one position early", V.scratch_entries,
     "for t in range(end + 1 - m, end + 1)])\n            Vb",
     "for t in range(end - m, end)])\n            Vb", _verify_all),
    ("root read from the raw rows", V.sequence_row, "if pos < L:", "if pos <= L:", _verify_all),
    ("path not reversed", V.path_to_root, "return path[::-1]", "return path", _verify_all),
    ("partial block compressed", C.compress_prefix, "0, L // m, m, g, store", "0, (L + m - 1) // m, m, g, store",
     _compress),
    ("bf16 rounding bit off by one", S._round_f64_to_bf16, "keep_lsb = (bits >> np.uint64(45))",
     "keep_lsb = (bits >> np.uint64(44))", _storage),
    ("capacity refused at an exact fit", R.refresh_commit_request, "if L + n > rawK.shape[0]:",
     "if L + n >= rawK.shape[0]:", _refresh),
    ("compressed capacity refused at an exact fit", R.refresh_commit_request,
     "if j >= CK.shape[0]:", "if j >= CK.shape[0] - 1:", _refresh),
    # acceptance ([TSD-V4] §4.1)
    ("highest-index matching child", A.accept_walk, "                nxt = c\n                break",
     "                nxt = c", _accept),
    ("draft compared with the child's own target", A.accept_walk,
     "int(draft[c]) == int(target[cur])", "int(draft[c]) == int(target[c])", _accept),
    ("node 1 never considered", A.accept_walk, "for c in range(1, D):", "for c in range(2, D):",
     _accept),
    ("bonus from the draft", A.accept_walk, "return len(path), path, int(target[cur])",
     "return len(path), path, int(draft[cur])", _accept),
    # refresh ([TSD-V4] §4.2)
    ("last accepted token never closes a block", R.refresh_commit_request,
     "for e in range(L, L + n):", "for e in range(L, L + n - 1):", _refresh),
    ("committed rows by path index", R.refresh_commit_request, "rawK[L + i] = to_f64(treeK[u])",
     "rawK[L + i] = to_f64(treeK[i])", _refresh),
    ("entry index one high", R.refresh_commit_request, "j = (e + 1) // m - 1", "j = (e + 1) // m",
     _refresh),
    # the round: the steps in order, per request ([TSD-V4] §4.1, §4.4)
    ("walk given draft and target swapped", RD.verify_round,
     "accept_walk(par, draft[b], target[b])", "accept_walk(par, target[b], draft[b])", _round),
    ("reported entry one block high", RD.verify_round, "                        j = (e + 1) // m - 1",
     "                        j = (e + 1) // m", _round),
    ("reported raw rows shifted", RD.verify_round, "raw_rows=(rK[Lb:L_new].copy(), rV[Lb:L_new].copy())",
     "raw_rows=(rK[Lb - 1:L_new - 1].copy(), rV[Lb - 1:L_new - 1].copy())", _round),
    ("another request's tree", RD.verify_round, "par = [int(x) for x in parents[b]]",
     "par = [int(x) for x in parents[0]]", _round),
    # indexer (the sparse C4 path)
    ("ties to the higher index", I.topk_ascending, "key=lambda j: (-float(scores[j]), j)",
     "key=lambda j: (-float(scores[j]), -j)", _indexer),
    ("one entry short", I.topk_ascending, "order[:k]", "order[:k - 1]", _indexer),
    ("list not ascending", I.topk_ascending, "return np.sort(np.asarray(order[:k], dtype=np.int32))",
     "return np.asarray(order[:k], dtype=np.int32)", _indexer),
    ("scores summed in fp64", I.index_scores, "s = (s + prod).astype(np.float32)",
     "s = s.astype(np.float64) + prod", _indexer),
    ("incomplete block selectable", I.indexer_select, "n4 = int(L) // 4", "n4 = (int(L) + 3) // 4",
     _indexer),
    # storage rounding
    ("bf16 ties rounded up", S._round_f64_to_bf16, "(bits + half_minus_one + keep_lsb)",
     "(bits + half_minus_one + np.uint64(1))", _storage),
    ("f64 storage rounded to f32", S.round_to_storage, "    if store == \"f64\":\n        return x.copy()",
     "    if store == \"f64\":\n        return x.astype(np.float32).astype(np.float64)", _storage),
    ("f32 storage not rounded", S.round_to_storage,
     "return x.astype(np.float32).astype(np.float64)", "return x.copy()", _storage),
]


@pytest.mark.parametrize("name,func,old,new,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(monkeypatch, name, func, old, new, pins):
    pin_list = pins()
    mutant = _mutant(func, old, new)
    _install(monkeypatch, func, mutant)
    assert any(_fails(pin) for pin in pin_list), f"no pin fails under: {name}"


CONTROLS = {}
for _name, _func, _old, _new, _pins in MUTANTS:
    CONTROLS.setdefault(_func, (_old, _pins))


@pytest.mark.parametrize("func", list(CONTROLS), ids=[f.__name__ for f in CONTROLS])
def test_rewriting_without_a_change_keeps_every_pin_passing(monkeypatch, func):
    # control: the same rewrite and installation with the text left as it is; every pin passes,
    # so a failure above comes from the planted mistake, not from the mechanism
    old, pins = CONTROLS[func]
    pin_list = pins()
    _install(monkeypatch, func, _mutant(func, old, old))
    failed = [i for i, pin in enumerate(pin_list) if _fails(pin)]
    assert not failed, f"{func.__name__}: pins {failed} fail without a change"
