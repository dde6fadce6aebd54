#!/usr/bin/env python
"""Benchmark of the DDTree tree-verify step on one GB300 (or N replicas).

A step is one pass of the whole hot path over one batch of synthetic input:
the verify of every layer of a 64-layer hybrid target (48 gated-DeltaNet
layers: 16 q/k heads, 48 v heads, dk = dv = 128; 16 full-attention layers:
24 query heads, 4 KV heads, head size 256, q8_0 cache of 32,768 tokens,
window 2048; pattern [GDN, GDN, GDN, attention] x 16), greedy acceptance over
a 151,936-entry vocabulary, and commit of the accepted path into every layer.
Budget 22 (a 22-node DDTree, top-4 expansion, depth <= 12); the target's
argmax is planted along the tree's deepest path (up to 8 nodes), so commit
moves a realistic accepted path.  The step is captured once in a CUDA graph
and replayed.

Metric: verified tree nodes per second per layer = B * N * 64 / step time,
plus the dominant kernel's fraction of the measured HBM roofline.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun each rank runs an independent replica on its own GPU (the
path has no exchange step); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "verified tree nodes/s per layer at budget 22, 32K ctx; % of HBM roofline"
UNIT = "nodes/s/layer"
N_LAYERS, N_GDN, N_ATTN = 64, 48, 16
ACCEPT_CHAIN = 16  # accept launches per timed replay, each over its own copy of the logits
BUDGET, VOCAB, CTX, WINDOW, PLANT = 22, 151936, 32768, 2048, 8
DRAFT_BLOCK, TOPK, TAU = 16, 4, 6.0   # draft positions per tree, expansion width, pruning margin
CLOCK_LOAD_S = 0.5                     # untimed replays of the step on each side of the timed steps, for the clock samples
GDN = synth.GDN_27B
ATT = synth.ATTN_27B
CONV = synth.CONV_27B
SEED = 1234 + 3
WORKLOAD = ("64-layer hybrid verify step: 48 gated-DeltaNet layers (16 qk / 48 v heads, dk=dv=128) + "
            "16 attention layers (24 q / 4 kv heads, D=256, q8_0 KV 32768 tokens, window 2048), "
            "22-node tree, accept over vocab 151936, commit")


def is_attn(layer):
    return layer % 4 == 3


# ---------------------------------------------------------------------------- inputs
MAX_REPLAYS = 512          # replays between resets that the cache capacity allows


def make_host_inputs(rng, n_layers=N_LAYERS, ctx=CTX):
    """Host-side inputs of the step (numpy), seeded; the first n_layers layers
    over a cache of ctx committed tokens."""
    par, tok = synth.ddtree(rng, BUDGET, VOCAB)
    parent, n_nodes = synth.batch_trees([par], BUDGET)
    tokens = tok[None].astype(np.int32)
    planted = synth.deepest_path(par)[:PLANT]
    logits = synth.random_logits(rng, 1, BUDGET, VOCAB)
    synth.plant_path(logits, tokens, planted)
    cap = ctx + BUDGET * MAX_REPLAYS + 64
    layers = []
    for layer in range(n_layers):
        if is_attn(layer):
            a = synth.attn_inputs(rng, 1, BUDGET, **ATT)
            a["cache"] = synth.kv_cache(rng, 1, ATT["Hkv"], cap, ATT["D"], synth.KV_Q8_0)
            layers.append(("attn", a))
        else:
            layers.append(("gdn", synth.gdn_inputs(rng, 1, BUDGET, **GDN)))
    # the short convolution in front of every GDN layer (measured beside the
    # step, not inside it); drawn from its own stream so the step's inputs
    # stay the same
    crng = np.random.default_rng(SEED + 7919)
    conv = [synth.conv_inputs(crng, 1, BUDGET, CONV["C"], CONV["K"]) for kind, _ in layers if kind == "gdn"]
    # the draft's logits for the next tree (its construction is measured beside the step)
    draft = synth.draft_logits(np.random.default_rng(SEED + 104729), 1, DRAFT_BLOCK, VOCAB)
    return dict(parent=parent, n_nodes=n_nodes, tokens=tokens, logits=logits, layers=layers, cap=cap, ctx=ctx,
                planted=planted, conv=conv, draft=draft)


def step_inputs(host):
    """The per-step inputs of a host input set, in the order the step's input
    buffer packs them: (name, array)."""
    out = [("parent", host["parent"]), ("n_nodes", host["n_nodes"]), ("tokens", host["tokens"]),
           ("logits", host["logits"])]
    for li, (kind, d) in enumerate(host["layers"]):
        keys = ("q", "k_new", "v_new") if kind == "attn" else ("q", "k", "v", "beta", "log_alpha")
        out += [(f"{li}.{k}", d[k]) for k in keys]
    return [(name, np.ascontiguousarray(a)) for name, a in out]


# ---------------------------------------------------------------------------- algorithmic bytes
def gdn_bytes(L=0):
    """One GDN verify with the previous step's accepted path of length L
    pending: the state is read, brought up to date and written back."""
    Hk, Hv, dk, dv, N = GDN["Hk"], GDN["Hv"], GDN["dk"], GDN["dv"], BUDGET
    state = Hv * dv * dk * 4 * (2 if L else 1)
    pend = L * (Hv * dv * 4 + Hv * 4 + Hk * dk * 2)
    qk = 2 * N * Hk * dk * 2
    v = N * Hv * dv * 2
    scal = 2 * N * Hv * 4
    out = N * Hv * dv * 4
    u = N * Hv * dv * 4
    g = N * Hv * 4
    kc = N * Hk * dk * 2
    return state + pend + qk + v + scal + out + u + g + kc


def attn_bytes():
    Hq, Hkv, D, N = ATT["Hq"], ATT["Hkv"], ATT["D"], BUDGET
    row = D + D // 32 * 2                      # q8_0: codes + fp16 scales per (token, head)
    kv = 2 * (WINDOW - 1) * Hkv * row          # visible cached keys and values
    q = N * Hq * D * 2
    out = N * Hq * D * 4
    new = 2 * N * Hkv * D * 2
    tree = 2 * 2 * N * Hkv * row               # tree slots written, then read
    return kv + q + out + new + tree


def conv_bytes():
    """One tree conv: x read, conv state read, taps read, output written."""
    C, K, N = CONV["C"], CONV["K"], BUDGET
    return N * C * 2 + (K - 1) * C * 2 + C * K * 4 + N * C * 4


def conv_commit_bytes(L):
    """Conv-state commit of all GDN layers: K-1 rows gathered from the state
    and the accepted inputs, K-1 rows written."""
    C, K = CONV["C"], CONV["K"]
    return N_GDN * 2 * (K - 1) * C * 2 if L else 0


def ddtree_bytes():
    """Tree construction: the draft's logits read once; top-K lists and the
    tree written."""
    return DRAFT_BLOCK * VOCAB * 4 + DRAFT_BLOCK * TOPK * 8 + BUDGET * 12 + 8


def accept_bytes():
    return BUDGET * VOCAB * 4


def commit_bytes(L):
    """Commit of the KV caches (the GDN states are committed inside the
    next step's verify)."""
    row = ATT["D"] + ATT["D"] // 32 * 2
    return N_ATTN * 2 * 2 * L * ATT["Hkv"] * row


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (200 ms period); only those stamped between
    mark() and stop() count, i.e. the samples taken while the GPU ran the
    timed steps and the same steps around them."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_mark = None

    def mark(self):
        self.t_mark = time.time()

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        t_stop = time.time()
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[9], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                ts = None
            if ts is not None and self.t_mark is not None and not (self.t_mark <= ts <= t_stop):
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------- peaks / profiles
def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_source_hash(kind):
    files = {"gdn": ["gdn_verify.cu"],
             "attn": ["attn_verify.cu", "attn_verify_tc.cu", "attn_common.cuh", "tcgen05.cuh", "cluster.cuh"],
             "accept": ["accept.cu"], "commit": ["commit.cu"], "conv": ["conv_tree.cu"], "conv_commit": ["conv_tree.cu"],
             "ddtree": ["ddtree.cu", "cluster.cuh"]}
    h = hashlib.sha256()
    for f in files[kind] + ["common.cuh", "tree.cuh"]:
        with open(os.path.join(ROOT, "speculative_decoding_tree_layer_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kind):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            t = json.load(f)
        e = t[kind]
        if e.get("source_hash") == kernel_source_hash(kind):
            return e.get("bytes_per_launch")
    except (OSError, KeyError, ValueError):
        pass
    return None


# ---------------------------------------------------------------------------- GPU step
class GpuStep:
    """Device buffers + the step's C-ABI calls (captured into a CUDA graph)."""

    def __init__(self, host, torch, dflv):
        self.torch, self.dflv = torch, dflv
        t = torch
        dev = "cuda"
        self.host = host
        cap = host["cap"]
        N = BUDGET
        self.ctx = host["ctx"]
        # ---- per-step inputs: one packed pinned host buffer and two device
        #      twins (the step of factor-set parity p reads twin p, so the next
        #      step's inputs can be copied in while a step runs)
        offs, total = {}, 0
        for name, a in step_inputs(host):
            total = (total + 255) // 256 * 256
            offs[name] = (total, a)
            total += a.nbytes
        self.offs = offs
        self.in_bytes = total
        self.h_in = t.empty(total, dtype=t.uint8, pin_memory=True)
        self.d_ins = [t.empty(total, dtype=t.uint8, device=dev) for _ in range(2)]
        self.load_inputs(host)

        def view_of(buf, name):
            o, a = offs[name]
            tdt = {np.dtype(np.uint16): t.int16, np.dtype(np.float32): t.float32,
                   np.dtype(np.int32): t.int32}[a.dtype]
            return buf[o:o + a.nbytes].view(tdt).view(*a.shape)

        self._view_of = view_of
        self.bound = 0

        def view(name):
            return view_of(self.d_ins[0], name)

        self.parent, self.n_nodes, self.tokens, self.logits = (view("parent"), view("n_nodes"), view("tokens"),
                                                               view("logits"))
        # ---- persistent state and outputs
        self.status = t.zeros(1, dtype=t.int32, device=dev)
        self.n_past = t.full((1,), self.ctx, dtype=t.int32, device=dev)
        self.path = t.zeros((1, N), dtype=t.int32, device=dev)
        self.path_len = t.zeros(1, dtype=t.int32, device=dev)
        self.next_token = t.zeros(1, dtype=t.int32, device=dev)
        self.best = t.zeros((1, N), dtype=t.int32, device=dev)
        self.h_out = t.empty((2, N + 2), dtype=t.int32, pin_memory=True)   # two slots: steps t and t+1
        # every layer but the first follows a kernel that writes neither its
        # committed state / cache prefix nor the tree: those may be read early
        early = dflv.DFLV_FLAG_EARLY_PREFETCH
        self.gdn_desc = dflv.gdn_desc(1, N, GDN["Hk"], GDN["Hv"], GDN["dk"], GDN["dv"])
        self.gdn_desc_next = dflv.gdn_desc(1, N, GDN["Hk"], GDN["Hv"], GDN["dk"], GDN["dv"], early)
        self.attn_desc = dflv.attn_desc(1, N, ATT["Hq"], ATT["Hkv"], ATT["D"], cap, WINDOW, dflv.DFLV_KV_Q8_0,
                                        1.0 / np.sqrt(ATT["D"]))
        self.attn_desc_next = dflv.attn_desc(1, N, ATT["Hq"], ATT["Hkv"], ATT["D"], cap, WINDOW, dflv.DFLV_KV_Q8_0,
                                             1.0 / np.sqrt(ATT["D"]), early)
        # one merge workspace for every attention layer (the calls are
        # ordered on one stream)
        self.attn_ws_bytes = dflv.dflv_attn_workspace_size(self.attn_desc)
        self.attn_ws = t.empty(max(self.attn_ws_bytes, 16), dtype=t.uint8, device=dev)
        self.layers = []
        self.states, self.factors, self.caches = [], [], []
        self.state0 = []
        for li, (kind, d) in enumerate(host["layers"]):
            if kind == "gdn":
                st = t.from_numpy(d["state"]).to(dev)
                L = dict(kind="gdn", q=view(f"{li}.q"), k=view(f"{li}.k"), v=view(f"{li}.v"),
                         beta=view(f"{li}.beta"), log_alpha=view(f"{li}.log_alpha"), state=st,
                         out=t.empty((1, N, GDN["Hv"], GDN["dv"]), device=dev),
                         u=[t.empty((1, N, GDN["Hv"], GDN["dv"]), device=dev) for _ in range(2)],
                         g=[t.empty((1, N, GDN["Hv"]), device=dev) for _ in range(2)],
                         kc=[t.empty((1, N, GDN["Hk"], GDN["dk"]), dtype=t.int16, device=dev) for _ in range(2)])
                # two factor sets: a step writes one and applies the other (deferred commit)
                L["fac"] = [dflv.gdn_factors(L["u"][i], L["g"][i], L["kc"][i]) for i in range(2)]
                self.states.append(st)
                self.state0.append(st.clone())
            else:
                c = d["cache"]
                dc = {k: t.from_numpy(v).to(dev) for k, v in c.items()}
                L = dict(kind="attn", q=view(f"{li}.q"), k_new=view(f"{li}.k_new"), v_new=view(f"{li}.v_new"),
                         out=t.empty((1, N, ATT["Hq"], ATT["D"]), device=dev), dc=dc,
                         kv=dflv.kv_layer(dc["kq"], dc["vq"], dc["ks"], dc["vs"]))
                self.caches.append(L["kv"])
            self.layers.append(L)
        self.launches_per_step = N_GDN + N_ATTN + 2 + 2  # accept and commit: two kernels each
        # ---- the short convolution of every GDN layer (measured beside the step)
        self.conv_desc = dflv.conv_desc(1, N, CONV["C"], CONV["K"])
        self.conv_desc_next = dflv.conv_desc(1, N, CONV["C"], CONV["K"], early)
        self.conv = []
        for d in host["conv"]:
            c = {k: t.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).to(dev) for k, v in d.items()}
            c["state0"] = c["state"].clone()
            c["out"] = t.empty((1, N, CONV["C"]), device=dev)
            self.conv.append(c)
        # ---- draft-tree construction (measured beside the step)
        self.draft = t.from_numpy(host["draft"]).to(dev)
        self.root_token = t.zeros(1, dtype=t.int32, device=dev)
        self.tree = dict(topk_tok=t.empty((1, DRAFT_BLOCK, TOPK), dtype=t.int32, device=dev),
                         topk_logp=t.empty((1, DRAFT_BLOCK, TOPK), device=dev),
                         parent=t.empty((1, N), dtype=t.int32, device=dev),
                         tokens=t.empty((1, N), dtype=t.int32, device=dev),
                         n_nodes=t.empty(1, dtype=t.int32, device=dev), score=t.empty((1, N), device=dev))
        self.ddtree_desc = dflv.ddtree_desc(1, DRAFT_BLOCK, VOCAB, TOPK, N, TAU)

    def load_inputs(self, host):
        """Packs a host input set of the same shapes into the pinned buffer
        and copies it to both device buffers the captured steps read."""
        hv = self.h_in.numpy()
        for name, a in step_inputs(host):
            o, a0 = self.offs[name]
            assert a.shape == a0.shape and a.dtype == a0.dtype, name
            hv[o:o + a.nbytes] = a.view(np.uint8).reshape(-1)
        for d in self.d_ins:
            d.copy_(self.h_in)

    def bind(self, which):
        """Points every per-step input of the calls at device buffer `which`."""
        v = lambda name: self._view_of(self.d_ins[which], name)
        self.parent, self.n_nodes, self.tokens, self.logits = v("parent"), v("n_nodes"), v("tokens"), v("logits")
        for li, L in enumerate(self.layers):
            keys = ("q", "k", "v", "beta", "log_alpha") if L["kind"] == "gdn" else ("q", "k_new", "v_new")
            for key in keys:
                L[key] = v(f"{li}.{key}")
        self.bound = which

    # one pass of the hot path: every layer's verify (the GDN layers first
    # commit the previous step's accepted path into their state: deferred
    # commit), acceptance, commit of the KV caches.  Step `par` writes
    # factor set par and applies set 1 - par.
    def gdn_verify(self, li, L, par):
        return self.dflv.dflv_tree_gdn_verify_pending(
            self.gdn_desc if li == 0 else self.gdn_desc_next, self.parent, self.n_nodes, L["q"], L["k"], L["v"],
            L["beta"], L["log_alpha"], L["state"], L["fac"][1 - par], self.path, self.path_len, L["out"],
            L["fac"][par], self.status)

    def attn_verify(self, L, desc=None):
        return self.dflv.dflv_tree_attn_verify(desc or self.attn_desc_next, self.parent, self.n_nodes, self.n_past,
                                               L["q"], L["k_new"], L["v_new"], L["kv"], L["out"], self.status,
                                               self.attn_ws, self.attn_ws_bytes)

    def step(self, par):
        dflv, chk = self.dflv, self.dflv.check
        for li, L in enumerate(self.layers):
            if L["kind"] == "gdn":
                chk(self.gdn_verify(li, L, par), "gdn verify")
            else:
                chk(self.attn_verify(L), "attn verify")
        chk(dflv.dflv_accept_greedy(1, BUDGET, VOCAB, self.logits, self.tokens, self.parent, self.n_nodes,
                                    self.path, self.path_len, self.next_token, self.best, self.status), "accept")
        chk(dflv.dflv_commit_rollback(None, 0, [], [], self.attn_desc, len(self.caches), self.caches, self.path,
                                      self.path_len, self.n_past, self.status), "commit")

    def reset(self):
        """Committed state back to its initial value (between passes)."""
        for s, s0 in zip(self.states, self.state0):
            s.copy_(s0)
        self.n_past.fill_(self.ctx)
        self.path_len.zero_()  # nothing pending
        for c in self.conv:
            c["state"].copy_(c["state0"])

    def conv_verify(self, i):
        c = self.conv[i]
        return self.dflv.dflv_tree_conv_verify(self.conv_desc if i == 0 else self.conv_desc_next, self.parent,
                                               self.n_nodes, c["x"], c["state"], c["w"], c["out"], self.status)

    def ddtree_build(self):
        tr = self.tree
        return self.dflv.dflv_ddtree_build(self.ddtree_desc, self.draft, self.root_token, tr["topk_tok"],
                                           tr["topk_logp"], tr["parent"], tr["tokens"], tr["n_nodes"], tr["score"],
                                           self.status)

    def conv_commit(self):
        return self.dflv.dflv_conv_commit(self.conv_desc, len(self.conv), [c["state"] for c in self.conv],
                                          [c["x"] for c in self.conv], self.path, self.path_len, self.status)


L2_FLUSH_BYTES = 2 * 129 * 2**20   # twice the L2


class L2Flush:
    """Writes a buffer twice the size of the L2 on the current stream, so
    that the next replay starts with none of its inputs cached."""

    def __init__(self, torch):
        self.buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")
        self.i = 0

    def __call__(self):
        self.i += 1
        self.buf.fill_(self.i)


def cold_replays(torch, graph, count, flush, stream):
    """Replays `graph` `count` times on `stream`, each after an L2 flush and
    between its own pair of CUDA events; returns the replay times in ms.
    The flush is still running when the events and the replay are submitted,
    so the host's submission stays off the measured interval."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(count)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            flush()
            a.record()
            graph.replay()
            b.record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def pct(xs):
    """p10 / p50 / p90 of a list of times."""
    return [float(np.percentile(xs, q)) for q in (10, 50, 90)]


def kernel_chain_ms(S, torch, stream, steps, warmup, flush):
    """Launch duration of each kernel kind inside its own chain, from cold
    L2: every replay follows an L2 flush.  The accept runs as a chain of
    ACCEPT_CHAIN launches, each over its own copy of the logits (together
    larger than the L2, so every launch reads cold logits), which spreads the
    replay's event and submission overhead like the verify chains; the other
    kinds with one launch per step are replayed as a graph of that one
    launch.  Returns (mean per launch, p10/p50/p90 per launch over the
    replays)."""
    dflv, chk = S.dflv, S.dflv.check
    logit_sets = [S.logits] + [S.logits.clone() for _ in range(ACCEPT_CHAIN - 1)]

    def gdn_chain():
        for li, L in enumerate(S.layers):
            if L["kind"] == "gdn":
                chk(S.gdn_verify(li, L, 0), "gdn verify")

    def attn_chain():
        for L in S.layers:
            if L["kind"] == "attn":
                chk(S.attn_verify(L), "attn verify")

    def accept(logits=None):
        chk(dflv.dflv_accept_greedy(1, BUDGET, VOCAB, S.logits if logits is None else logits, S.tokens, S.parent,
                                    S.n_nodes, S.path, S.path_len, S.next_token, S.best, S.status), "accept")

    def accept_chain():
        for lg in logit_sets:
            accept(lg)

    def commit():
        chk(dflv.dflv_commit_rollback(None, 0, [], [], S.attn_desc, len(S.caches), S.caches, S.path, S.path_len,
                                      S.n_past, S.status), "commit")

    def conv_chain():
        for i in range(len(S.conv)):
            chk(S.conv_verify(i), "conv verify")

    def conv_commit():
        chk(S.conv_commit(), "conv commit")

    def ddtree():
        chk(S.ddtree_build(), "ddtree build")

    out, dist = {}, {}
    for name, fn, n in (("gdn", gdn_chain, N_GDN), ("attn", attn_chain, N_ATTN), ("accept", accept_chain, ACCEPT_CHAIN),
                        ("commit", commit, 1), ("conv", conv_chain, N_GDN), ("conv_commit", conv_commit, 1),
                        ("ddtree", ddtree, 1)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        S.reset()
        with torch.cuda.stream(stream):
            accept()  # an accepted path: the GDN verifies apply it as their pending commit
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                g.replay()
        torch.cuda.synchronize()
        ts = cold_replays(torch, g, steps, flush, stream)
        out[name] = float(np.sum(ts)) / (steps * n)
        dist[name] = [x / n for x in pct(ts)]
        S.reset()
        torch.cuda.synchronize()
    del logit_sets
    return out, dist


# ---------------------------------------------------------------------------- at scale
# The long-context, wide-tree stress shapes: 8 sequences with 64-node trees,
# one attention layer over a 131,072-token q4_0 cache with full attention
# (24 query / 4 KV heads, D = 256) and one GDN layer of the 27B shape.
SCALE_B, SCALE_N, SCALE_CTX = 8, 64, 131072


SCALE_ATTN = ((synth.KV_Q4_0, 8), (synth.KV_Q4_0, 22), (synth.KV_Q4_0, 64), (synth.KV_TQ3_0, 64))


def scale_bytes_attn(N=SCALE_N, kv=synth.KV_Q4_0):
    """Attention at the stress shape: every cached key and value read once,
    q read, o written, the tree's new K/V read and its slots written and read."""
    Hq, Hkv, D, B, P = ATT["Hq"], ATT["Hkv"], ATT["D"], SCALE_B, SCALE_CTX
    code = D // 32 * 12 if kv == synth.KV_TQ3_0 else D // 2
    row = code + D // 32 * 2                   # codes + fp16 scales per (token, head)
    kv = B * 2 * P * Hkv * row
    return kv + B * N * (Hq * D * 2 + Hq * D * 4 + 2 * Hkv * D * 2) + B * 2 * 2 * N * Hkv * row


def scale_flops_attn(N=SCALE_N):
    """Q K^T and P V over every (node, query head, visible key): 2 * 2 * D
    flops each (the kernel's hi/lo operand split adds passes, not counted)."""
    Hq, D, B, P = ATT["Hq"], ATT["D"], SCALE_B, SCALE_CTX
    return 2 * 2 * D * B * N * Hq * (P + N)


def bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured sustained"
    except (OSError, KeyError, ValueError):
        return 1700.0, "fallback sustained"


def scale_bytes_gdn():
    Hk, Hv, dk, dv, B, N = GDN["Hk"], GDN["Hv"], GDN["dk"], GDN["dv"], SCALE_B, SCALE_N
    return B * (Hv * dv * dk * 4 + 2 * N * Hk * dk * 2 + N * Hv * dv * 2 + 2 * N * Hv * 4 + 2 * N * Hv * dv * 4 +
                N * Hv * 4 + N * Hk * dk * 2)


def scale_trees(torch, n=SCALE_N):
    """The stress shapes' trees: SCALE_B DDTree-shaped trees of n nodes."""
    rng = np.random.default_rng(SEED + 37 + (n if n != SCALE_N else 0))
    pars = [synth.ddtree(rng, n, VOCAB)[0] for _ in range(SCALE_B)]
    parent, n_nodes = synth.batch_trees(pars, n)
    return torch.from_numpy(parent).to("cuda"), torch.from_numpy(n_nodes).to("cuda")


def dev_bf16(torch, g, *shape, unit=False):
    """N(0, 1) bf16 bits on the device (L2-normalised over the last axis if
    `unit`, as q and k of a GDN layer are)."""
    x = torch.randn(*shape, generator=g, device="cuda")
    if unit:
        x = x / x.norm(dim=-1, keepdim=True)
    return x.to(torch.bfloat16).view(torch.int16)


def scale_gdn_set(torch, dflv, g):
    """One GDN layer's inputs, state and outputs at the stress shape."""
    B, N, dev = SCALE_B, SCALE_N, "cuda"
    Hk, Hv, dk, dv = GDN["Hk"], GDN["Hv"], GDN["dk"], GDN["dv"]
    u, gg = torch.empty(B, N, Hv, dv, device=dev), torch.empty(B, N, Hv, device=dev)
    kc = torch.empty(B, N, Hk, dk, dtype=torch.int16, device=dev)
    return dict(
        u=u, g=gg, kc=kc,
        st=torch.randn(B, Hv, dv, dk, generator=g, device=dev) * 0.02,
        q=dev_bf16(torch, g, B, N, Hk, dk, unit=True), k=dev_bf16(torch, g, B, N, Hk, dk, unit=True),
        v=dev_bf16(torch, g, B, N, Hv, dv),
        beta=torch.sigmoid(torch.randn(B, N, Hv, generator=g, device=dev)),
        la=-torch.nn.functional.softplus(torch.randn(B, N, Hv, generator=g, device=dev)),
        o=torch.empty(B, N, Hv, dv, device=dev),
        fac=dflv.gdn_factors(u, gg, kc))


def scale_measure(torch, dflv, flush, reps=8, rounds=10):
    """Per-launch time of the attention and GDN verify at the stress shapes,
    `reps` launches back to back per graph (early prefetch after the first),
    each replay after an L2 flush.  Attention reads 1.2 GB per launch, so its
    launches share one set of buffers; the GDN launches rotate over `reps`
    input sets so that none reads what the one before left in the L2.  Inputs
    are drawn on the device from a seeded generator."""
    dev = "cuda"
    g = torch.Generator(device=dev)
    g.manual_seed(SEED + 31)
    B, N, P = SCALE_B, SCALE_N, SCALE_CTX
    Hq, Hkv, D = ATT["Hq"], ATT["Hkv"], ATT["D"]
    cap = P + N
    out = {}
    par_d, nn_d = scale_trees(torch)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream()

    def bf16(*shape, unit=False):
        return dev_bf16(torch, g, *shape, unit=unit)

    def timed(fn):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn(0)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            for r in range(reps):
                fn(r)
        with torch.cuda.stream(stream):
            for _ in range(3):
                graph.replay()
        torch.cuda.synchronize()
        return float(np.sum(cold_replays(torch, graph, rounds, flush, stream))) / (rounds * reps)

    # attention, full attention over a 131,072-token cache: the budget sweep
    # over q4_0 (8 nodes: below the ridge, HBM-bound; 22 and 64: tensor-bound)
    # and the TQ3_0 cache at 64 nodes
    tpk, tkind = bf16_peak()
    n_past = torch.full((B,), P, dtype=torch.int32, device=dev)
    for kvt in (synth.KV_Q4_0, synth.KV_TQ3_0):
        code = D // 32 * 12 if kvt == synth.KV_TQ3_0 else D // 2
        kq = torch.randint(0, 256, (B, Hkv, cap, code), generator=g, device=dev, dtype=torch.uint8)
        vq = torch.randint(0, 256, (B, Hkv, cap, code), generator=g, device=dev, dtype=torch.uint8)
        ks = (torch.rand(B, Hkv, cap, D // 32, generator=g, device=dev) * 0.02).to(torch.float16).view(torch.int16)
        vs = (torch.rand(B, Hkv, cap, D // 32, generator=g, device=dev) * 0.02).to(torch.float16).view(torch.int16)
        kv = dflv.kv_layer(kq, vq, ks, vs)
        for kind, Nn in SCALE_ATTN:
            if kind != kvt:
                continue
            par_n, nn_n = scale_trees(torch, Nn)
            q, kn, vn = bf16(B, Nn, Hq, D), bf16(B, Nn, Hkv, D), bf16(B, Nn, Hkv, D)
            o = torch.empty((B, Nn, Hq, D), device=dev)
            descs = [dflv.attn_desc(B, Nn, Hq, Hkv, D, cap, 0, kvt, 1.0 / np.sqrt(D), f)
                     for f in (0, dflv.DFLV_FLAG_EARLY_PREFETCH)]
            wsb = dflv.dflv_attn_workspace_size(descs[0])
            ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)

            def attn(r):
                # every launch attends at the same position: n_past does not
                # move, and the tree's slots are rewritten in place
                dflv.check(dflv.dflv_tree_attn_verify(descs[r > 0], par_n, nn_n, n_past, q, kn, vn, kv, o,
                                                      status, ws, wsb))

            ms = timed(attn)
            byt, flops = scale_bytes_attn(Nn, kvt), scale_flops_attn(Nn)
            tf = flops / (ms * 1e-3) / 1e12
            gbs = byt / (ms * 1e-3) / 1e9
            name = f"attn_{'tq3' if kvt == synth.KV_TQ3_0 else 'q4'}_131k_b8_n{Nn}"
            out[name] = {"ms_per_launch": ms, "nodes_per_s_per_layer": B * Nn / (ms * 1e-3),
                         "algorithmic_bytes_per_launch": byt, "achieved": gbs, "unit": "GB/s",
                         "flop_per_byte": flops / byt,
                         "algorithmic_flops_per_launch": flops, "tflops": tf,
                         "tensor_peak_tflops": tpk, "tensor_frac": tf / tpk,
                         "tensor_peak_source": tkind + " bf16_tflops",
                         "bound": "hbm" if flops / byt < tpk * 1e12 / (hbm_peak()[0] * 1e9) else "tensor"}
            del q, kn, vn, o, ws
        del kq, vq, ks, vs, kv
    # GDN: 27B shape, batch 8, 64-node trees
    Hk, Hv, dk, dv = GDN["Hk"], GDN["Hv"], GDN["dk"], GDN["dv"]
    sets = [scale_gdn_set(torch, dflv, g) for _ in range(reps)]
    gdescs = [dflv.gdn_desc(B, N, Hk, Hv, dk, dv, f) for f in (0, dflv.DFLV_FLAG_EARLY_PREFETCH)]

    def gdn(r):
        d = sets[r]
        dflv.check(dflv.dflv_tree_gdn_verify(gdescs[r > 0], par_d, nn_d, d["q"], d["k"], d["v"], d["beta"], d["la"],
                                             d["st"], d["o"], d["fac"], status))

    ms = timed(gdn)
    byt = scale_bytes_gdn()
    out["gdn_b8_n64"] = {"ms_per_launch": ms, "nodes_per_s_per_layer": B * N / (ms * 1e-3),
                         "algorithmic_bytes_per_launch": byt,
                         "achieved": byt / (ms * 1e-3) / 1e9, "unit": "GB/s"}
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    return out


def capture_step(S, torch, stream):
    """Eager warm-up of the step on the capture stream (sets kernel
    attributes once), reset, then one CUDA graph per step parity (the factor
    sets alternate between steps).  Returns the two graphs; the state is
    reset, so the first replay has nothing pending."""
    with torch.cuda.stream(stream):
        S.step(0)
        S.step(1)
    torch.cuda.synchronize()
    S.reset()
    torch.cuda.synchronize()
    graphs = [torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()]
    for par in range(2):
        S.bind(par)  # the step of parity par reads input buffer par
        with torch.cuda.graph(graphs[par], stream=stream):
            S.step(par)
    S.bind(0)
    torch.cuda.synchronize()
    assert int(S.status.item()) == 0, f"device status {int(S.status.item())}"
    return graphs


def run_gpu(args, rank, world):
    import torch

    import speculative_decoding_tree_layer_gb300 as dflv

    dflv.load()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    rng = np.random.default_rng(SEED + rank)
    host = make_host_inputs(rng)
    S = GpuStep(host, torch, dflv)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    graphs = capture_step(S, torch, stream)
    count = [0]

    def replay():
        graphs[count[0] % 2].replay()
        count[0] += 1


    # ---- device-resident timing
    S.reset()
    count[0] = 0
    for _ in range(args.warmup):
        replay()
    torch.cuda.synchronize()
    barrier(world)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x for x in vis.split(",") if x.strip().isdigit()]
    clocks = ClockSampler(int(ids[local]) if local < len(ids) else local)
    clocks.start()
    time.sleep(0.3)

    def load_for(seconds, max_replays):
        # the same step, replayed untimed, so that the clock samples around
        # the short timed region are taken under its load; at most
        # max_replays, which the cache capacity allows between rewinds
        t, n = time.perf_counter(), 0
        while time.perf_counter() - t < seconds and n + 32 <= max_replays:
            for _ in range(32):
                replay()
            n += 32
            torch.cuda.synchronize()

    def rewind():
        # every replay commits its accepted path and so advances the cache
        # position; the phases below start again at the context length (the
        # window keeps each step's work the same at any position)
        S.n_past.fill_(S.ctx)

    clocks.mark()
    load_for(CLOCK_LOAD_S, MAX_REPLAYS - args.warmup - 1)
    rewind()
    torch.cuda.synchronize()
    barrier(world)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        replay()
    t1.record()
    torch.cuda.synchronize()
    barrier(world)
    ms = t0.elapsed_time(t1)
    rewind()
    load_for(CLOCK_LOAD_S, MAX_REPLAYS - 1)
    clk = clocks.stop()
    status = int(S.status.item())
    L = int(S.path_len.item())
    assert status == 0, f"device status {status}"
    ms_max = reduce_max(world, ms)

    # ---- the spread over steps: the same replays, each between its own events
    rewind()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in evs:
        a.record()
        replay()
        b.record()
    torch.cuda.synchronize()
    step_pct = pct([a.elapsed_time(b) for a, b in evs])

    # ---- per-kernel durations: every kernel kind of the step launched back
    #      to back as in the step (all its layers, same buffers, same launch
    #      overlap), one CUDA graph per kind, each replay after an L2 flush and
    #      between its own events on the launching stream; per launch =
    #      chain time / launches
    flush = L2Flush(torch)
    per, dist = kernel_chain_ms(S, torch, stream, args.steps, args.warmup, flush)
    status = int(S.status.item())
    assert status == 0, f"device status {status} after the per-kernel chains"
    scale = scale_measure(torch, dflv, flush) if not args.no_scale else {}
    del flush
    # ---- end to end: pinned host inputs -> device, step, result -> host, every
    #      step, through the same captured C-ABI calls.  The step of parity p
    #      reads device input buffer p, so step t+1's inputs are copied on a
    #      second stream straight into its buffer while step t runs (the copy
    #      engines work beside the SMs), once step t-1 has finished reading
    #      that buffer.  The accepted path goes to one of two pinned host
    #      slots; the host reads step t's path once step t+1 is enqueued, so
    #      its wait overlaps the next step (the path feeds the host's output,
    #      not the next step's inputs, which the device produces), and the
    #      last step's path is read inside the timed region.
    S.reset()
    count[0] = 0
    copy_stream = torch.cuda.Stream()
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    read_done = [torch.cuda.Event(), torch.cuda.Event()]
    result = [torch.cuda.Event(), torch.cuda.Event()]
    torch.cuda.synchronize()

    def e2e_steps(n):
        t0 = count[0]  # replay() alternates the parity from here
        with torch.cuda.stream(copy_stream):
            S.d_ins[t0 % 2].copy_(S.h_in, non_blocking=True)
            copied[t0 % 2].record(copy_stream)
        for t in range(n):
            par = (t0 + t) % 2
            if t + 1 < n:
                with torch.cuda.stream(copy_stream):
                    if t >= 1:
                        copy_stream.wait_event(read_done[1 - par])  # step t-1 read that buffer
                    S.d_ins[1 - par].copy_(S.h_in, non_blocking=True)   # the next step's inputs
                    copied[1 - par].record(copy_stream)
            slot = S.h_out[t % 2]
            with torch.cuda.stream(stream):
                stream.wait_event(copied[par])
                replay()
                read_done[par].record(stream)
                slot[: BUDGET].copy_(S.path[0], non_blocking=True)
                slot[BUDGET].copy_(S.path_len[0], non_blocking=True)
                slot[BUDGET + 1].copy_(S.next_token[0], non_blocking=True)
                result[t % 2].record(stream)
            if t > 0:                         # the host reads the previous step's accepted path
                result[(t - 1) % 2].synchronize()
                _ = int(S.h_out[(t - 1) % 2, BUDGET])
        if n > 0:
            result[(n - 1) % 2].synchronize()
            _ = int(S.h_out[(n - 1) % 2, BUDGET])

    e2e_steps(args.warmup)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_steps(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    status = int(S.status.item())
    assert status == 0, f"device status {status} after the end-to-end steps"
    e2e_ms = reduce_max(world, e0.elapsed_time(e1))
    d2h = (BUDGET + 2) * 4
    return dict(ms=ms_max, per=per, dist=dist, step_pct=step_pct, scale=scale, clocks=clk, L=L, e2e_ms=e2e_ms, h2d=S.in_bytes, d2h=d2h,
                launches=S.launches_per_step, dev_name=torch.cuda.get_device_name(), host=host)


# ---------------------------------------------------------------------------- CPU oracle
def oracle_block_sample(host, parts=None):
    """The oracle on one [GDN, GDN, GDN, attention] block of the step plus
    accept and commit of that block: returns seconds.  With a list `parts`,
    appends the seconds of each part (GDN verify of the three layers,
    attention verify, accept, commit)."""
    import oracle

    parent, n_nodes = host["parent"], host["n_nodes"]
    gdn_layers = [d for kind, d in host["layers"][:4] if kind == "gdn"]
    a = host["layers"][3][1]
    cache = synth.copy_cache(a["cache"])   # the sample's own cache, outside the timed parts
    t0 = time.perf_counter()
    for d in gdn_layers:
        oracle.tree_gdn_verify(parent, n_nodes, d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], d["state"])
    t1 = time.perf_counter()
    oracle.tree_attn_verify(parent, n_nodes, np.array([CTX], np.int32), a["q"], a["k_new"], a["v_new"], cache,
                            WINDOW, oracle.KV_Q8_0)
    t2 = time.perf_counter()
    path, plen, _, _ = oracle.accept_greedy(host["logits"], host["tokens"], parent, n_nodes)
    t3 = time.perf_counter()
    for d in gdn_layers:
        oracle.gdn_commit(d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], path, plen, d["state"])
    oracle.kv_commit(cache, oracle.KV_Q8_0, path, plen, np.array([CTX], np.int32))
    t4 = time.perf_counter()
    if parts is not None:
        parts.append((t1 - t0, t2 - t1, t3 - t2, t4 - t3))
    return t4 - t0


def oracle_c4_sequence():
    """The oracle on one sequence of the long-context stress shape at 22
    nodes: attention over a 131,072-token q4_0 cache with full attention,
    and one GDN layer; returns (attention seconds, GDN seconds)."""
    import oracle

    rng = np.random.default_rng(SEED + 41)
    parent, n_nodes = synth.batch_trees([synth.ddtree(rng, BUDGET, VOCAB)[0]], BUDGET)
    inp = synth.attn_inputs(rng, 1, BUDGET, ATT["Hq"], ATT["Hkv"], ATT["D"])
    cache = synth.kv_cache(rng, 1, ATT["Hkv"], SCALE_CTX + BUDGET, ATT["D"], synth.KV_Q4_0)
    g = synth.gdn_inputs(rng, 1, BUDGET, **GDN)
    t0 = time.perf_counter()
    oracle.tree_attn_verify(parent, n_nodes, np.array([SCALE_CTX], np.int32), inp["q"], inp["k_new"],
                            inp["v_new"], cache, 0, oracle.KV_Q4_0)
    t1 = time.perf_counter()
    oracle.tree_gdn_verify(parent, n_nodes, g["q"], g["k"], g["v"], g["beta"], g["log_alpha"], g["state"])
    return t1 - t0, time.perf_counter() - t1


def cpu_baseline(host, min_seconds=3.0, min_reps=3):
    """The oracle on all host cores (its loops over independent (sequence,
    head) and output rows run in parallel), and on one thread: samples
    repeated for at least `min_seconds` and `min_reps`, median reported."""
    import oracle

    oracle.build()
    cores = os.cpu_count() or 1
    res = {}
    parts = []
    for threads in (cores, 1):
        used = oracle.set_threads(threads)
        ts, t0 = [], time.perf_counter()
        while len(ts) < min_reps or time.perf_counter() - t0 < min_seconds:
            ts.append(oracle_block_sample(host, parts if threads == cores else None))
        res[threads] = (used, float(np.median(ts)), len(ts))
    oracle.set_threads(cores)
    used, t, n = res[cores]
    gdn_s, attn_s, acc_s, com_s = (float(np.median([p[j] for p in parts])) for j in range(4))
    per_layer = {"gdn": BUDGET / (gdn_s / 3), "attn": BUDGET / attn_s, "unit": "nodes/s per layer",
                 "accept_seconds": acc_s, "commit_seconds": com_s,
                 "what": "the parts of the all-core sample: one GDN layer (3 per block) and one attention layer "
                         "at the step's shapes"}
    try:
        c4_attn, c4_gdn = oracle_c4_sequence()
        c4 = {"attn_seconds": c4_attn, "gdn_seconds": c4_gdn, "attn_nodes_per_s": BUDGET / c4_attn,
              "gdn_nodes_per_s": BUDGET / c4_gdn, "cores": used,
              "what": "one sequence at 22 nodes of the long-context stress shape (131,072-token q4_0 cache, "
                      "full attention) on all cores; the stress shape has 8 sequences: x8 the time is an "
                      "extrapolation, not a measurement"}
    except Exception as e:  # a baseline that cannot run is reported, not fatal
        c4 = {"error": f"{type(e).__name__}: {e}"}
    return {"value": BUDGET * 4 / t, "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"one [GDN, GDN, GDN, attention] block of the step (4 of 64 layers) + accept over the "
                      f"full vocab + commit of that block; C oracle, fp64, parallel over (sequence, head) and "
                      f"output rows; median of {n} samples",
            "seconds_per_sample": t, "samples": n,
            "single_thread": {"value": BUDGET * 4 / res[1][1], "cores": 1, "seconds_per_sample": res[1][1],
                              "samples": res[1][2]},
            "per_layer": per_layer, "long_context_one_sequence": c4}


# ---------------------------------------------------------------------------- distributed plumbing
def init_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if os.environ.get("BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def reduce_max(world, x):
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(world, steps, ms_max):
    """Whole-job throughput: every rank verified BUDGET nodes through N_LAYERS
    layers per step; the slowest rank's time bounds the job."""
    return world * BUDGET * N_LAYERS * steps / (ms_max * 1e-3)


# ---------------------------------------------------------------------------- profiling mode
def profile_one(kind, launches):
    """One kernel of the step on its own workload (the first layer of that
    kind, or accept / commit of one step), launched back to back."""
    import torch

    import speculative_decoding_tree_layer_gb300 as dflv

    dflv.load()
    torch.cuda.set_device(0)
    if kind == "gdn_scale":
        # the GDN verify at the stress shape (8 sequences, 64-node trees)
        g = torch.Generator(device="cuda")
        g.manual_seed(SEED + 31)
        par_d, nn_d = scale_trees(torch)
        d = scale_gdn_set(torch, dflv, g)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        desc = dflv.gdn_desc(SCALE_B, SCALE_N, GDN["Hk"], GDN["Hv"], GDN["dk"], GDN["dv"])
        for _ in range(launches):
            dflv.check(dflv.dflv_tree_gdn_verify(desc, par_d, nn_d, d["q"], d["k"], d["v"], d["beta"], d["la"],
                                                 d["st"], d["o"], d["fac"], status))
        torch.cuda.synchronize()
        print(json.dumps({"kernel": kind, "launches": launches, "status": int(status.item())}))
        return
    rng = np.random.default_rng(SEED)
    host = make_host_inputs(rng, n_layers=4)
    S = GpuStep(host, torch, dflv)
    li, L = next((i, L) for i, L in enumerate(S.layers) if L["kind"] == ("attn" if kind == "attn" else "gdn"))
    if kind in ("conv", "conv_commit", "ddtree"):
        S.step(1)
        torch.cuda.synchronize()
        for _ in range(launches):
            dflv.check(S.conv_verify(0) if kind == "conv" else S.conv_commit() if kind == "conv_commit"
                       else S.ddtree_build())
        torch.cuda.synchronize()
        print(json.dumps({"kernel": kind, "launches": launches, "status": int(S.status.item())}))
        return
    # one step first: both factor sets written and an accepted path pending
    S.step(1)
    S.n_past.fill_(CTX)
    for _ in range(launches):
        if kind == "gdn":
            dflv.check(S.gdn_verify(li, L, 0))
        elif kind == "attn":
            dflv.check(S.attn_verify(L, S.attn_desc))
        elif kind == "accept":
            dflv.check(dflv.dflv_accept_greedy(1, BUDGET, VOCAB, S.logits, S.tokens, S.parent, S.n_nodes, S.path,
                                               S.path_len, S.next_token, S.best, S.status))
        else:
            S.step(0)
            S.n_past.fill_(CTX)
    torch.cuda.synchronize()
    print(json.dumps({"kernel": kind, "launches": launches, "status": int(S.status.item())}))


# ---------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-scale", action="store_true", help="skip the at-scale kernel measurements")
    ap.add_argument("--kernel", choices=["gdn", "attn", "accept", "commit", "conv", "conv_commit", "ddtree",
                                         "gdn_scale"],
                    default=None,
                    help="profiling mode: launch one kernel of the step --launches times on its "
                         "single-layer workload and exit (for ncu captures)")
    ap.add_argument("--launches", type=int, default=3)
    args = ap.parse_args()
    if args.kernel:
        return profile_one(args.kernel, args.launches)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "ours" and args.steps + args.warmup + 1 > MAX_REPLAYS:
        ap.error(f"--steps + --warmup must stay below {MAX_REPLAYS} (KV cache capacity)")
    rank, world = init_dist()

    if args.impl == "reference":
        if rank != 0:
            return
        rng = np.random.default_rng(SEED)
        host = make_host_inputs(rng, n_layers=4)
        import oracle

        oracle.build()
        cores = oracle.set_threads(os.cpu_count() or 1)
        for _ in range(args.warmup):
            oracle_block_sample(host)
        ts = [oracle_block_sample(host) for _ in range(args.steps)]
        t = float(np.sum(ts))
        value = BUDGET * 4 * args.steps / t
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * t / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic",
                "config": {"workload": WORKLOAD + " (bounded sample per step: one 4-layer block + accept + commit)",
                           "batch": 1, "budget": BUDGET, "ctx": CTX, "window": WINDOW, "kv": "q8_0"},
                "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                                 "sample": "per step: one [GDN, GDN, GDN, attention] block + accept + commit; "
                                           "parallel over (sequence, head) and output rows"},
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    r = run_gpu(args, rank, world)
    peak, peak_kind = hbm_peak()
    per = r["per"] or {}
    L = r["L"]
    ab = dict(gdn=gdn_bytes(L), attn=attn_bytes(), accept=accept_bytes(), commit=commit_bytes(L),
              conv=conv_bytes(), conv_commit=conv_commit_bytes(L), ddtree=ddtree_bytes())
    launches = dict(gdn=N_GDN, attn=N_ATTN, accept=1, commit=1)
    step_mb = sum(ab[k] * launches[k] for k in launches) / 1e6
    # dominant kernel: the largest share of the step
    shares = {k: per[k] * launches[k] for k in per if k in launches} if per else {}
    beside = {}
    for k in ("conv", "conv_commit", "ddtree"):
        if per.get(k):
            gbs = ab[k] / (per[k] * 1e-3) / 1e9
            beside[k] = {"ms_per_launch": per[k], "algorithmic_bytes_per_launch": ab[k], "achieved": gbs,
                         "unit": "GB/s", "frac": gbs / peak,
                         "launches": N_GDN if k == "conv" else 1}
    if "ddtree" in beside:
        beside["ddtree"]["launches"] = 1
        beside["ddtree"]["kernels_per_launch"] = 2
    dom = max(shares, key=shares.get) if shares else "commit"
    dur_ms = per.get(dom)
    achieved = ab[dom] / (dur_ms * 1e-3) / 1e9 if dur_ms else None
    value = aggregate_value(world, args.steps, r["ms"])
    e2e_value = aggregate_value(world, args.steps, r["e2e_ms"])
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16/f32 (q8_0 KV)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": 1, "budget": BUDGET, "ctx": CTX, "window": WINDOW,
                   "kv": "q8_0", "vocab": VOCAB, "accepted_len": L,
                   "l2": f"inputs larger than L2 (~{step_mb:.0f} MB touched per step); no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "device": r["dev_name"]},
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": (achieved / peak) if achieved else None,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": ab[dom],
                     "avg_launch_ms": dur_ms,
                     "launch_timing": "one replay = the chain of all launches of this kernel in the step, "
                                      "back to back (accept: 16 launches, each over its own copy of the "
                                      "logits; one launch for the other kernels launched once per step); each "
                                      "replay after an L2 flush (a buffer twice the L2 written) and between "
                                      "its own CUDA events on the launching stream; mean over the replays",
                     "traffic": profiled_traffic(dom)},
        "kernels_ms_per_launch": per,
        "kernels_ms_per_launch_p10_p50_p90": r["dist"],
        "step_ms_p10_p50_p90": r["step_pct"],
        "nodes_per_s_per_layer": {"step": value / world,
                                  **{k: BUDGET / (per[k] * 1e-3) for k in ("gdn", "attn") if per.get(k)}},
        "at_scale": {"what": "the stress shapes beside the step: 8 sequences; attention over a 131,072-token "
                             "cache with full attention, q4_0 at 8, 22 and 64 nodes per tree and TQ3_0 at 64; GDN "
                             "of the 27B shape at 64 nodes; 8 launches back to back per CUDA graph (the GDN "
                             "launches on 8 distinct input sets), an L2 flush before each replay, CUDA events",
                     **{k: dict(v, peak=peak, frac=v["achieved"] / peak) for k, v in r["scale"].items()}},
        "beside_the_step": {"what": "the short convolution in front of each GDN layer (48 tree-conv launches "
                                    "back to back, C=10240, K=4), the commit of its window (one launch, 48 "
                                    "layers) and the construction of the next draft tree from the draft's "
                                    "logits (16 positions x 151936, top-4, budget 22, tau 6: a top-K/log-sum-exp "
                                    "kernel and a best-first kernel); timed like the step's kernels, not part "
                                    "of the step",
                            **beside},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "how": "every step: the step's inputs from pinned host memory, copied on a second stream while "
                       "the previous step runs straight into the device buffer its captured calls read (two "
                       "buffers, one captured graph per step parity), one replay of the captured C-ABI calls of "
                       "the step, the accepted path copied to pinned host memory; the host reads step t's path "
                       "once step t+1 is enqueued (two host slots), and the last step's path inside the timed "
                       "region"},
        "gpu_launches": r["launches"] * args.steps,
        "clocks": r["clocks"],
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(r["host"])
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
