"""GPU parity for candidate-tree drafts and tree-mask block verification
(Alignment Drift App. E.3: the drafter's ranked tokens fill a fixed tree, the
target verifies every node in one pass under a tree attention mask, the
longest root path that matches the target's argmax is accepted; a
one-branch tree reproduces the linear decoder):

  * one tree verify on the fp32 tiny model against the oracle's tree verify,
    acceptance along a branch that is not the first child, and the commit of
    that path checked through the next draft and the next verify;
  * whole tree decodes against the oracle's tree decode, round by round;
  * large-v3 bf16: the one-branch tree gives the linear decoder's rounds and
    transcript bit for bit, and the 11-row tree gives the autoregressive
    transcript.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import model as M
from gpu_common import MARGIN_BF16, dev_i32, logits_close

pytestmark = pytest.mark.gpu

# 11 candidate rows under the anchor: the top three tokens at depth 1, the
# first one's argmax chain down to depth 8, one more row under the second.
TREE_PARENT = [-1, 0, 0, 0, 1, 2, 4, 6, 7, 8, 9, 10]
TREE_RANK = [0, 0, 1, 2, 0, 0, 0, 0, 0, 0, 0, 0]


@pytest.fixture(scope="module")
def RB():
    import __graft_entry__ as g
    g.build()
    from speculative_whisper_asr_gb300 import binding, runtime
    return runtime, binding


def _stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.fixture(scope="module")
def tiny(RB):
    R, B = RB
    s = synth.TINY
    tw = synth.target_weights(s, 0)
    dw = synth.drafter_weights(s, 0, tw)
    A = synth.encoder_states(s, 0, 0)
    orc = M.Oracle(s, tw, dw)
    dec = R.Decoder(s, tw, dw, max_batch=1, max_frames=1500, max_block=len(TREE_PARENT))
    req = dec.slots([0])
    dec.cross_kv(req, dec.enc_tensor(A), [1500])
    dec.set_tree(TREE_PARENT, TREE_RANK)
    return s, tw, dw, A, orc, dec, req


def test_tiny_tree_verify_accept_commit_vs_oracle(RB, tiny):
    """The greedy continuation y1, y2 sits on rows 2 and 5 (the second
    depth-1 branch); every other row holds a wrong token.  The tree verify's
    logits match the oracle's for all 12 rows, acceptance walks 0 -> 2 -> 5
    and emits y1, y2, y3, and after the commit the next draft and the next
    one-token verify match the oracle's (the path's keys, values and history
    rows sit at positions L+1, L+2)."""
    R, B = RB
    s, tw, dw, A, orc, dec, req = tiny
    N = len(TREE_PARENT)
    ref = M.greedy_cached(orc, orc.new_request(A), 8).tokens
    rng = np.random.default_rng(7)
    toks = [int(t) for t in rng.integers(0, 50000, size=N)]
    for j in range(1, N):
        while toks[j] in ref[:4]:
            toks[j] = (toks[j] + 1) % 50000
    toks[0], toks[2], toks[5] = ref[0], ref[1], ref[2]
    b = dec.new_batch(req, [64])
    b.prefill()
    assert b.transcripts()[0] == ref[:1]
    dec.draft(req, b.block, 0.0, 0, 0, b.q_logits)     # a round's draft folds the prompt rows into the history
    b.tblock[0, :N] = dev_i32(toks)
    b.blen[0] = N
    lg = torch.empty(1, N, s.vocab, device="cuda")
    B.ws_verify_tree(dec.ctx, 1, req.data_ptr(), N, b.tblock.data_ptr(), b.blen.data_ptr(), b.ttarget.data_ptr(),
                     lg.data_ptr(), _stream())
    r = orc.new_request(A)
    M.prefill(orc, r, 64)
    ora = orc.verify_tree(r, toks, TREE_PARENT)
    logits_close(lg[0].cpu().numpy(), ora, 1e-4)
    g = b.ttarget[0, :N].tolist()
    assert g == lg[0].argmax(dim=1).tolist()
    assert g == [M.argmax_lowest(z) for z in ora]
    a = b._args(B.WS_ACCEPT_TREE, N, b.tblock, b.blen, b.ttarget, b.block, b.blen)
    B.ws_accept(dec.ctx, 1, req.data_ptr(), a, _stream())
    acc, path = M.accept_tree(toks, TREE_PARENT, g, 63, s.eos_id)
    assert path == [0, 2, 5] and acc.emitted == ref[1:4]
    assert int(b.n_acc[0]) == 2 and b.transcripts()[0] == ref[:4]
    orc.commit_path(r, path)
    r.L += 1 + acc.a
    assert int(dec.lengths(req)[0]) == r.L
    anchor = ref[3]
    assert int(b.block[0, 0]) == anchor
    dec.draft(req, b.block, 0.0, 0, 0, b.q_logits)
    logits_close(b.q_logits[0].cpu().numpy(), orc.draft_logits(r, anchor), 1e-4)
    lg1 = torch.empty(1, 1, s.vocab, device="cuda")
    t1 = torch.zeros(1, 1, dtype=torch.int32, device="cuda")
    dec.verify(req, dev_i32([[anchor]]), dev_i32([1]), t1, lg1)
    logits_close(lg1[0].cpu().numpy(), orc.verify(r, [anchor]), 1e-4)
    assert dec.status() == 0


def test_tiny_tree_decode_matches_oracle_round_by_round(RB, tiny):
    """Whole tree decodes (40 tokens): per round, the tree's tokens, the
    accepted count and the emitted tokens equal the oracle's; the transcript
    equals the oracle's tree decode and its autoregressive greedy decode.  A
    round whose drafter ranks, or the target argmax of a row on its accepted
    path, sit within 1e-4 (relative) of a tie ends the comparison."""
    R, B = RB
    s, tw, dw, A, orc, dec, req = tiny
    N = len(TREE_PARENT)
    budget = 40
    log = []
    ref = M.speculative_greedy_tree(orc, orc.new_request(A), budget, TREE_PARENT, TREE_RANK, log)
    assert ref.tokens == M.greedy_cached(orc, orc.new_request(A), budget).tokens
    b = dec.new_batch(req, [budget])
    b.prefill()
    rounds = 0
    while b.poll_done() < 1:
        b.spec_step(rounds + 1, tree=True, graph=False)
        q, toks, lg, path = log[rounds]
        n = len(toks)
        tied = False
        for j in range(1, n):        # ranked drafter tokens near a tie
            row = np.sort(q[M_depth(j) - 1])[::-1]
            k = TREE_RANK[j]
            gaps = [row[k] - row[k + 1]] + ([row[k - 1] - row[k]] if k > 0 else [])
            if min(gaps) < 1e-4 * max(abs(row[k]), 1.0):
                tied = True
        for z in lg[path]:               # the target rows the walk compares against
            top = np.sort(z)[-2:]
            if top[1] - top[0] < 1e-4 * max(abs(top[1]), 1.0):
                tied = True
        if tied:
            break
        assert b.tblock[0, :n].tolist() == toks, rounds
        assert int(b.n_acc[0]) == ref.accepted[rounds], rounds
        rounds += 1
    else:
        assert rounds == ref.rounds
        assert b.transcripts()[0] == ref.tokens
    assert rounds >= min(ref.rounds, 4)
    assert dec.status() == 0


def M_depth(j):
    d = 0
    while TREE_PARENT[j] >= 0:
        j = TREE_PARENT[j]
        d += 1
    return d


def test_large_v3_chain_tree_is_linear_and_tree_equals_autoregressive(RB):
    """Large-v3 bf16 batch 1, 96 tokens.  The one-branch tree (a chain of K
    rows taking each mask row's argmax) runs exactly the linear decoder's
    computation: the same accepted counts every round and the same
    transcript, bit for bit.  The 11-row tree gives the autoregressive
    transcript."""
    R, B = RB
    s = synth.LARGE_V3
    tw = synth.target_weights(s, 1)
    dw = synth.drafter_weights(s, 1, tw)
    A = synth.encoder_states(s, 1, 0)
    dec = R.Decoder(s, tw, dw, max_batch=1, max_frames=1500, max_block=len(TREE_PARENT))
    req = dec.slots([0])
    dec.cross_kv(req, dec.enc_tensor(A), [1500])
    b = dec.new_batch(req, [96])
    R.run_ar(dec, b)
    ar = b.transcripts()[0]

    def accepted_per_round(tree):
        bb = dec.new_batch(req, [96], draft_logits=True)
        bb.prefill()
        acc = []
        while bb.poll_done() < 1:
            bb.spec_step(len(acc) + 1, tree=tree)
            acc.append(int(bb.n_acc[0]))
        return acc, bb.transcripts()[0]

    lin_acc, lin = accepted_per_round(False)
    dec.set_tree([-1] + list(range(s.K)), [0] * (s.K + 1))
    chain_acc, chain = accepted_per_round(True)
    assert chain_acc == lin_acc and chain == lin == ar
    dec.set_tree(TREE_PARENT, TREE_RANK)
    tree_acc, tree = accepted_per_round(True)
    assert tree == ar
    print(f"rounds: linear {len(lin_acc)}, tree {len(tree_acc)}; "
          f"rounds with a >= 1: linear {sum(a > 0 for a in lin_acc)}, tree {sum(a > 0 for a in tree_acc)}")
    dec.set_tree()
    assert dec.status() == 0


def test_large_v3_bf16_tree_verify_branch_commit_vs_oracle(RB):
    """The bf16 tensor-core attention under a tree mask: large-v3, the
    oracle's greedy continuation on rows 2 and 5, random tokens elsewhere.
    All 12 rows' logits match the oracle's tree verify (2e-2), acceptance
    walks 0 -> 2 -> 5, and after the commit the next draft and the next
    one-token verify match the oracle's (2e-2)."""
    R, B = RB
    s = synth.LARGE_V3
    tw = synth.target_weights(s, 1)
    dw = synth.drafter_weights(s, 1, tw)
    A = synth.encoder_states(s, 1, 0)
    N = len(TREE_PARENT)
    orc = M.Oracle(s, tw, dw)
    r = orc.new_request(A)
    acc0, lg0 = M.prefill(orc, r, 64)
    y0 = acc0.next_anchor
    y1 = M.argmax_lowest(orc.verify(r, [y0])[0]); r.L += 1
    y2 = M.argmax_lowest(orc.verify(r, [y1])[0]); r.L -= 1
    rng = np.random.default_rng(11)
    toks = [int(t) for t in rng.integers(0, 50000, size=N)]
    for j in range(1, N):
        while toks[j] in (y0, y1, y2):
            toks[j] = (toks[j] + 1) % 50000
    toks[0], toks[2], toks[5] = y0, y1, y2
    dec = R.Decoder(s, tw, dw, max_batch=1, max_frames=1500, max_block=N)
    req = dec.slots([0])
    dec.cross_kv(req, dec.enc_tensor(A), [1500])
    dec.set_tree(TREE_PARENT, TREE_RANK)
    b = dec.new_batch(req, [64])
    b.prefill()
    b.block[0, 0] = y0                                    # the oracle's first token is the anchor
    dec.draft(req, b.block, 0.0, 0, 0, b.q_logits)
    b.tblock[0, :N] = dev_i32(toks)
    b.blen[0] = N
    lg = torch.empty(1, N, s.vocab, device="cuda")
    B.ws_verify_tree(dec.ctx, 1, req.data_ptr(), N, b.tblock.data_ptr(), b.blen.data_ptr(), b.ttarget.data_ptr(),
                     lg.data_ptr(), _stream())
    ora = orc.verify_tree(r, toks, TREE_PARENT)
    logits_close(lg[0].cpu().numpy(), ora, 2e-2)
    g_o = [M.argmax_lowest(z) for z in ora]
    acc, path = M.accept_tree(toks, TREE_PARENT, g_o, 63, s.eos_id)
    assert path == [0, 2, 5]
    for j in path:                                         # the walk's decisions are not near ties
        assert M.top2_margin(ora[j]) > MARGIN_BF16
    a = b._args(B.WS_ACCEPT_TREE, N, b.tblock, b.blen, b.ttarget, b.block, b.blen)
    B.ws_accept(dec.ctx, 1, req.data_ptr(), a, _stream())
    assert int(b.n_acc[0]) == 2
    assert b.transcript[0, 1:4].tolist() == acc.emitted
    orc.commit_path(r, path)
    r.L += 1 + acc.a
    anchor = acc.next_anchor
    dec.draft(req, b.block, 0.0, 0, 0, b.q_logits)
    logits_close(b.q_logits[0].cpu().numpy(), orc.draft_logits(r, anchor), 2e-2)
    lg1 = torch.empty(1, 1, s.vocab, device="cuda")
    t1 = torch.zeros(1, 1, dtype=torch.int32, device="cuda")
    dec.verify(req, dev_i32([[anchor]]), dev_i32([1]), t1, lg1)
    logits_close(lg1[0].cpu().numpy(), orc.verify(r, [anchor]), 2e-2)
    assert dec.status() == 0
