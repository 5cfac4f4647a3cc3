"""Planted mistakes: each plausible error in an oracle must fail one of its pins.

Every test swaps one oracle function for a copy with a single mistake (on the
CPU, inside the oracle only) and runs the pin that should catch it; the pin
must raise.  This is the evidence that the pins constrain the oracle rather
than restate it.
"""
import numpy as np
import pytest

import test_oracle_attention as TA
import test_oracle_dta as TD
import test_oracle_logprob as TL
import test_oracle_trie as TT
import test_partition as TP
from oracle import attention as OA
from oracle import dta as OD
from oracle import logprob as OL
from oracle import mask as OM
from oracle import partition as OP
from oracle import trie as OT


# ------------------------------------------------------------ attention
def test_missing_scale_is_caught(monkeypatch):
    orig = OA.forward
    monkeypatch.setattr(OA, "forward", lambda q, k, v, mask, scale=None: orig(q, k, v, mask, 1.0))
    with pytest.raises(AssertionError):
        TA.test_single_sequence_equals_causal_sdpa()


def _forward_head_map_mod(q, k, v, mask, scale=None):
    """The forward with query head h reading kv head h % Hkv."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    o = np.zeros_like(q)
    lse = np.empty((Hq, T))
    for h in range(Hq):
        kv = h % Hkv
        s = scale * (q[:, h, :] @ k[:, kv, :].T)
        p, lse[h] = OA._softmax_rows(s, mask)
        o[:, h, :] = p @ v[:, kv, :]
    return o, lse


def test_wrong_head_map_is_caught(monkeypatch):
    monkeypatch.setattr(OA, "forward", _forward_head_map_mod)
    with pytest.raises(AssertionError):
        TA.test_single_sequence_equals_causal_sdpa()


def _backward_variant(drop_d=False, overwrite_dv=False):
    def bwd(q, k, v, o, do, mask, scale=None):
        T, Hq, d = q.shape
        g = Hq // k.shape[1]
        scale = 1.0 / np.sqrt(d) if scale is None else scale
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        for h in range(Hq):
            kv = h // g
            s = scale * (q[:, h, :] @ k[:, kv, :].T)
            p, _ = OA._softmax_rows(s, mask)
            if overwrite_dv:
                dv[:, kv, :] = p.T @ do[:, h, :]
            else:
                dv[:, kv, :] += p.T @ do[:, h, :]
            dp = do[:, h, :] @ v[:, kv, :].T
            D = 0.0 if drop_d else (do[:, h, :] * o[:, h, :]).sum(axis=-1)[:, None]
            ds = p * (dp - D)
            dq[:, h, :] = scale * (ds @ k[:, kv, :])
            dk[:, kv, :] += scale * (ds.T @ q[:, h, :])
        return dq, dk, dv
    return bwd


@pytest.mark.parametrize("mistake", ["drop_d", "overwrite_dv"])
def test_backward_mistakes_are_caught(monkeypatch, mistake):
    monkeypatch.setattr(OA, "backward", _backward_variant(**{mistake: True}))
    with pytest.raises(AssertionError):
        TA.test_backward_equals_autograd_dense_mask()


# ------------------------------------------------------------ trie and mask
def test_mask_off_by_one_is_caught(monkeypatch):
    orig = OM.mask_rows

    def strict(packed, r0, r1):              # j < i instead of j <= i
        rows = orig(packed, r0, r1)
        for i in range(r0, r1):
            rows[i - r0, i] = False
        return rows
    monkeypatch.setattr(OM, "mask_rows", strict)
    with pytest.raises(AssertionError):
        TT.test_worked_example_compressed()


def test_compression_without_sequence_check_is_caught(monkeypatch):
    def compress_any_chain(trie):
        stack = list(trie.root.children.values())
        while stack:
            node = stack.pop()
            while len(node.children) == 1:
                (child,) = node.children.values()
                node.tokens.extend(child.tokens)
                node.children = child.children
                for grandchild in node.children.values():
                    grandchild.parent = node
            stack.extend(node.children.values())
    monkeypatch.setattr(OT, "compress", compress_any_chain)
    with pytest.raises(AssertionError):
        TT.test_brute_force_pairs_exhaustive()


def test_exit_off_by_one_is_caught(monkeypatch):
    orig = OT.layout

    def layout_exit_short(trie, block=128, pad_to=None):
        p = orig(trie, block, pad_to)
        p.node_exit = p.node_exit - 1
        return p
    monkeypatch.setattr(OT, "layout", layout_exit_short)
    with pytest.raises(AssertionError):
        TT.test_worked_example_compressed()


# ------------------------------------------------------------ log-prob gather
def test_transition_from_the_wrong_row_is_caught(monkeypatch):
    def transition(self, pred_pos, label_pos):
        return float(self._row(label_pos - 1)[0][self.packed.token_ids[label_pos]])
    monkeypatch.setattr(OL._Gather, "transition", transition)
    with pytest.raises(AssertionError):
        TL.test_unpack_invariant_random_tries()


def test_internal_label_off_by_one_is_caught(monkeypatch):
    def internal(self, start, end):
        tok = self.packed.token_ids
        return np.array([self._row(p)[0][tok[p]] for p in range(start, end)])
    monkeypatch.setattr(OL._Gather, "internal", internal)
    with pytest.raises(AssertionError):
        TL.test_unpack_invariant_random_tries()


def test_entropy_sign_is_caught(monkeypatch):
    orig = OL.row_stats

    def flipped(row):
        lse, ent, mn, mx = orig(row)
        return lse, -ent, mn, mx
    monkeypatch.setattr(OL, "row_stats", flipped)
    with pytest.raises(AssertionError):
        TL.test_unpack_invariant_random_tries()


def test_predecessor_at_the_parent_start_is_caught(monkeypatch):
    def pred_parent_start(packed):
        pred = np.full(packed.T_pad, -1, np.int32)
        for j in range(packed.T_pad):
            n = int(packed.token_node[j])
            if n < 0:
                continue
            if j > int(packed.node_start[n]):
                pred[j] = j - 1
            elif int(packed.node_parent[n]) >= 0:
                pred[j] = int(packed.node_start[int(packed.node_parent[n])])
        return pred
    monkeypatch.setattr(OL, "token_pred", pred_parent_start)
    with pytest.raises(AssertionError):
        TL.test_brute_force_predecessors_exhaustive_pairs()


def _gather_backward_variant(mistake):
    """The gather backward with one mistake."""
    def bwd(logits, packed, grads):
        x = np.asarray(logits, dtype=np.float64)
        out = np.zeros_like(x)
        tok = packed.token_ids
        for sid, (g_lp, g_ent) in grads.items():
            for t, (p, lab) in enumerate(OL.sequence_pairs(packed, sid)):
                lq = OL.log_softmax(x[p])
                q = np.exp(lq)
                row = lab if mistake == "label_row" else p
                if g_lp is not None:
                    if mistake != "no_softmax_term":
                        out[row] -= g_lp[t] * q
                    out[row, tok[lab]] += g_lp[t]
                if g_ent is not None:
                    h = -(q * lq).sum()
                    sign = -1.0 if mistake == "entropy_sign" else 1.0
                    out[row] -= g_ent[t] * q * (lq + sign * h)
        return out
    return bwd


@pytest.mark.parametrize("mistake", ["label_row", "no_softmax_term", "entropy_sign"])
def test_gather_backward_mistakes_are_caught(monkeypatch, mistake):
    monkeypatch.setattr(OL, "gather_packed_tree_backward", _gather_backward_variant(mistake))
    with pytest.raises(AssertionError):
        TL.test_backward_equals_autograd_of_unpacked_sequences()
    with pytest.raises(AssertionError):
        TL.test_backward_closed_forms()


def test_unmodified_gather_backward_variant_passes(monkeypatch):
    monkeypatch.setattr(OL, "gather_packed_tree_backward", _gather_backward_variant(None))
    TL.test_backward_equals_autograd_of_unpacked_sequences()
    TL.test_backward_closed_forms()


def test_backward_without_transitions_is_caught(monkeypatch):
    orig = OL.sequence_pairs
    monkeypatch.setattr(OL, "sequence_pairs", lambda packed, sid: [
        (p, l) for p, l in orig(packed, sid) if l == p + 1])
    with pytest.raises(AssertionError):
        TL.test_backward_equals_autograd_of_unpacked_sequences()


def test_lm_head_without_transpose_is_caught(monkeypatch):
    monkeypatch.setattr(OL, "lm_head_logits", lambda hidden, weight: (
        np.asarray(hidden, dtype=np.float64) @ np.asarray(weight, dtype=np.float64)))
    with pytest.raises(AssertionError):
        TL.test_lm_head_logits_exact_products()


# ------------------------------------------------------------ DTA schedule
def test_shallowest_first_order_is_caught(monkeypatch):
    monkeypatch.setattr(OD, "greedy_order", lambda nodes, depth, packed: sorted(
        nodes, key=lambda n: (int(depth[n]), int(packed.node_entry[n]))))
    with pytest.raises(AssertionError):
        TD.test_worked_example_schedules()


def _schedule_variant(push_leaf_last=False, backward_first=False):
    def schedule(packed, chunk=2048):
        kids, top = OD.children(packed)
        depth = OD.depth_tokens(packed, kids)
        ops = []

        def visit(n):
            segs = OD.chunks(packed, n, chunk)
            leaf = not kids[n]
            pushed = segs if (push_leaf_last or not leaf) else segs[:-1]
            for t0, t1 in pushed:
                ops.append((OD.FWD_PUSH, t0, t1))
            if leaf and not push_leaf_last:
                ops.append((OD.FWD_BWD, *segs[-1]))
            if backward_first:
                for t0, t1 in reversed(pushed):
                    ops.append((OD.BWD_POP, t0, t1))
            for c in OD.greedy_order(kids[n], depth, packed):
                visit(c)
            if not backward_first:
                for t0, t1 in reversed(pushed):
                    ops.append((OD.BWD_POP, t0, t1))
        for n in OD.greedy_order(top, depth, packed):
            visit(n)
        return ops
    return schedule


@pytest.mark.parametrize("mistake", ["push_leaf_last", "backward_first"])
def test_schedule_mistakes_are_caught(monkeypatch, mistake):
    monkeypatch.setattr(OD, "schedule", _schedule_variant(**{mistake: True}))
    with pytest.raises(AssertionError):
        TD.test_worked_example_schedules()
    with pytest.raises(AssertionError):
        TD.test_structure_random_tries(3)


def test_unmodified_schedule_variant_passes(monkeypatch):
    # the copy used above, without a mistake, passes the same pins
    monkeypatch.setattr(OD, "schedule", _schedule_variant())
    TD.test_worked_example_schedules()
    TD.test_structure_random_tries(3)


# ------------------------------------------------------------ partitioner
def test_tree_tokens_without_sharing_is_caught(monkeypatch):
    monkeypatch.setattr(OP, "tree_tokens", lambda group: sum(len(s) for s in group))
    with pytest.raises(AssertionError):
        TP.test_tree_tokens_worked_example()


def test_dp_that_forgets_the_last_segment_is_caught(monkeypatch):
    def optimal_drop_last(seqs, n_groups):
        order = OP.dfs_order(seqs)
        n = len(order)
        inf = float("inf")
        best = [[inf] * (n + 1) for _ in range(n_groups + 1)]
        best[0][0] = 0
        for k in range(1, n_groups + 1):
            for j in range(1, n + 1):
                for i in range(k - 1, j):
                    if best[k - 1][i] == inf:
                        continue
                    c = OP.tree_tokens([seqs[order[t]] for t in range(i, j)])
                    best[k][j] = min(best[k][j], best[k - 1][i] if k > 1 else c)
        return int(min(best[k][n] for k in range(1, n_groups + 1)))
    monkeypatch.setattr(OP, "optimal_contiguous", optimal_drop_last)
    with pytest.raises(AssertionError):
        TP.test_optimal_contiguous_equals_exhaustive_enumeration()
