"""Checks of a GPU greedy verify against the oracle, shared by the GPU tests.

Where every row that decides a stream's outcome (rows 0..accept_len of the
stream) has an oracle top-1 fp32 margin above 1e-3, accept_len and next_token
must equal the oracle's bit for bit.  Where one of them is a near-tie,
several outcomes are correct, and the check accepts exactly those: the
GPU's per-row argmax ids (from lmhead_argmax on the same inputs) must each be
within 1e-3 of their row's oracle maximum for rows 0..accept_len, the drafts
must equal those ids before accept_len and differ from it at accept_len
(unless every draft was accepted), and next_token must be the id at
accept_len.
"""
import numpy as np

MARGIN = 1e-3


def near_best(logits_row, ids_all, tok):
    """Whether token `tok` is a candidate of the row whose oracle logit is
    within MARGIN of the row's maximum."""
    j = np.nonzero(ids_all == int(tok))[0]
    return j.size == 1 and float(logits_row[j[0]]) >= float(logits_row.max()) - MARGIN


def check_verify(res, drafts, acc_gpu, nxt_gpu, a_gpu, n_draft, n_streams, vm=None):
    """res: the oracle's VerifyResult; drafts [n_streams][n_draft]; acc_gpu,
    nxt_gpu [n_streams] from the GPU verify; a_gpu [T] GPU argmax ids of the
    same rows (required: the near-tie check is stated in terms of them)."""
    assert a_gpu is not None
    rows_per = n_draft + 1
    drafts = np.asarray(drafts, np.int64).reshape(n_streams, n_draft)
    acc_gpu = np.asarray(acc_gpu).reshape(-1)
    nxt_gpu = np.asarray(nxt_gpu).reshape(-1)
    a_gpu = np.asarray(a_gpu).reshape(-1)
    ids_all = np.arange(res.logits.shape[1]) if vm is None else np.asarray(vm)
    # per-row argmax ids: exact where the row's margin allows, else near-best
    for t in range(len(res.a)):
        if res.margin[t] > MARGIN:
            assert int(a_gpu[t]) == int(res.a[t]), (t, int(a_gpu[t]), int(res.a[t]))
        else:
            assert near_best(res.logits[t], ids_all, a_gpu[t]), (t, int(a_gpu[t]))
    for s in range(n_streams):
        r0 = s * rows_per
        acc = int(res.accept_len[s])
        ag = int(acc_gpu[s])
        if all(res.margin[t] > MARGIN for t in range(r0, r0 + acc + 1)):
            assert ag == acc, (s, ag, acc)
            assert int(nxt_gpu[s]) == int(res.next_token[s]), (s, int(nxt_gpu[s]), int(res.next_token[s]))
            continue
        # a near-tie decides: the GPU's outcome must be one of the correct ones
        assert 0 <= ag <= n_draft, (s, ag)
        for i in range(ag + 1):
            assert near_best(res.logits[r0 + i], ids_all, a_gpu[r0 + i]), (s, i, int(a_gpu[r0 + i]))
        for i in range(ag):
            assert int(drafts[s, i]) == int(a_gpu[r0 + i]), (s, i)
        if ag < n_draft:
            assert int(drafts[s, ag]) != int(a_gpu[r0 + ag]), (s, ag)
        assert int(nxt_gpu[s]) == int(a_gpu[r0 + ag]), (s, int(nxt_gpu[s]), int(a_gpu[r0 + ag]))
