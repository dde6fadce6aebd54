"""GPU parity of the benchmarked step as a whole.

The step that the benchmark times (bench.GpuStep, captured by
bench.capture_step into one CUDA graph per factor-set parity) is replayed on
a reduced stack and compared after every step with the oracle's eager step:
verify of every layer, greedy acceptance, commit of the accepted path into
every GDN state and KV cache ("Luce DFlash" README, "How it works": per-step
rollback leaves the committed prefix as if only the accepted tokens had been
decoded).

What the reduced stack keeps from the benchmark: the [GDN, GDN, GDN,
attention] pattern (two blocks), the 27B-class shapes, a 22-node DDTree,
a q8_0 cache with window 2048, early prefetch from the second layer on
(GDN -> attention -> GDN hand-offs included), the deferred commit (every GDN
verify applies the previous step's accepted path while it streams the
state), the KV-only commit kernel, and the captured graphs themselves.  Each
step copies fresh inputs (a new tree, new q/k/v, new logits with a planted
path of a different length) into the buffer the graphs read, so the pending
path of each step comes from a real accept of a different tree.
"""
import os
import sys

import numpy as np
import pytest
import torch

import synth
from gpu_util import assert_close, host

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

N_LAYERS, CTX, STEPS = 8, 4096, 3


@pytest.fixture(scope="module")
def dflv():
    import speculative_decoding_tree_layer_gb300 as pkg

    pkg.build()
    pkg.load()
    return pkg


def fresh_step_inputs(rng, host0, plant_len):
    """The per-step inputs of host0's shapes, drawn anew: a DDTree of the
    budget, its tokens, logits with the first plant_len nodes of the deepest
    path planted (0: no planting), and every layer's q/k/v (+ beta, log alpha)."""
    N, V = bench.BUDGET, bench.VOCAB
    par, tok = synth.ddtree(rng, N, V)
    parent, n_nodes = synth.batch_trees([par], N)
    tokens = tok[None].astype(np.int32)
    logits = synth.random_logits(rng, 1, N, V)
    if plant_len:
        synth.plant_path(logits, tokens, synth.deepest_path(par)[:plant_len])
    layers = []
    for kind, d in host0["layers"]:
        if kind == "attn":
            layers.append(("attn", synth.attn_inputs(rng, 1, N, **bench.ATT)))
        else:
            layers.append(("gdn", synth.gdn_inputs(rng, 1, N, **bench.GDN, state=False)))
    return dict(host0, parent=parent, n_nodes=n_nodes, tokens=tokens, logits=logits, layers=layers)


def test_benchmarked_step_matches_oracle(dflv, orc):
    rng = np.random.default_rng(4242)
    host0 = bench.make_host_inputs(rng, n_layers=N_LAYERS, ctx=CTX)
    S = bench.GpuStep(host0, torch, dflv)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    graphs = bench.capture_step(S, torch, stream)

    # the oracle's committed state: GDN states, caches, P
    ref_states = {li: d["state"].copy() for li, (kind, d) in enumerate(host0["layers"]) if kind == "gdn"}
    ref_caches = {li: synth.copy_cache(d["cache"]) for li, (kind, d) in enumerate(host0["layers"]) if kind == "attn"}
    P = CTX
    plants = [bench.PLANT, 0, 5]          # a long path, (almost surely) the root alone, a medium path
    lengths = []
    for t in range(STEPS):
        inp = fresh_step_inputs(rng, host0, plants[t])
        S.load_inputs(inp)
        with torch.cuda.stream(stream):
            graphs[t % 2].replay()
        torch.cuda.synchronize()
        assert int(S.status.item()) == 0, f"step {t}: device status {int(S.status.item())}"

        parent, n_nodes = inp["parent"], inp["n_nodes"]
        # ---- verify of every layer against the oracle's committed state
        for li, (kind, d) in enumerate(inp["layers"]):
            L = S.layers[li]
            if kind == "gdn":
                # the state the step verified against: the previous step's
                # accepted path applied (written back by the deferred commit)
                assert_close(host(L["state"]), ref_states[li], what=f"step {t} layer {li} state")
                ref = orc.tree_gdn_verify(parent, n_nodes, d["q"], d["k"], d["v"], d["beta"], d["log_alpha"],
                                          ref_states[li])
            else:
                ref = orc.tree_attn_verify(parent, n_nodes, np.array([P], np.int32), d["q"], d["k_new"],
                                           d["v_new"], ref_caches[li], bench.WINDOW, synth.KV_Q8_0)
            assert_close(host(L["out"])[0], ref[0], what=f"step {t} layer {li} ({kind}) out")
        # ---- acceptance: bit-exact
        rp, rl, rn, rb = orc.accept_greedy(inp["logits"], inp["tokens"], parent, n_nodes)
        Lg = int(host(S.path_len)[0])
        assert Lg == rl[0], f"step {t}: path length {Lg} vs {rl[0]}"
        assert np.array_equal(host(S.path)[0, :Lg], rp[0, :Lg])
        assert int(host(S.next_token)[0]) == rn[0]
        assert np.array_equal(host(S.best)[0], rb[0])
        lengths.append(Lg)
        # ---- the oracle commits eagerly
        for li, (kind, d) in enumerate(inp["layers"]):
            if kind == "gdn":
                ref_states[li] = orc.gdn_commit(d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], rp, rl,
                                                ref_states[li])
            else:
                orc.kv_commit(ref_caches[li], synth.KV_Q8_0, rp, rl, np.array([P], np.int32))
        P += int(rl[0])
        # ---- the KV caches after the step's commit: every committed slot bit-exact
        assert int(host(S.n_past)[0]) == P
        for li, ref_c in ref_caches.items():
            dc = S.layers[li]["dc"]
            for key in ("kq", "vq", "ks", "vs"):
                got = host(dc[key], ref_c[key].dtype)
                assert np.array_equal(got[:, :, :P], ref_c[key][:, :, :P]), f"step {t} layer {li} {key}"

    # ---- the last step's accepted path is still pending in the GDN states:
    #      bring copies up to date with the commit kernel and compare
    li_gdn = [li for li, L in enumerate(S.layers) if L["kind"] == "gdn"]
    copies = [S.layers[li]["state"].clone() for li in li_gdn]
    n_past = torch.zeros(1, dtype=torch.int32, device="cuda")
    dflv.check(dflv.dflv_commit_rollback(S.gdn_desc, len(li_gdn), copies,
                                         [S.layers[li]["fac"][(STEPS - 1) % 2] for li in li_gdn], None, 0, [],
                                         S.path, S.path_len, n_past, S.status))
    torch.cuda.synchronize()
    assert int(S.status.item()) == 0
    for li, c in zip(li_gdn, copies):
        assert_close(host(c), ref_states[li], what=f"layer {li} state after the last commit")
    # the inputs exercised more than the root-only path
    assert max(lengths) > 1, lengths
