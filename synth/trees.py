"""Seeded prefetching trees and their flat (CSR) layout.

The tree follows the prefetching tree of "PreSTO: Predictive Subtree Prefetching
for Fast LLM Power Sampling" (section 3.2, step (1), and Appendix C.1):

* the root v0 holds the current state and has cut index c0 = T (Example 2);
* expanding a node v creates an acceptance child v+ (which carries the request
  (v+, c) with a freshly drawn cut c) and a rejection child v- (which keeps the
  state of v and, as Figure 8(b) labels it, the cut of v);
* a request is feasible when c <= cut(v) (Condition 1); an infeasible request
  is deferred, keeps its cut, and v+ is not expanded, while v- is still
  enqueued;
* BFS stops when N_pf feasible requests are collected or the queue is empty.

Every feasible request becomes one *segment* of scored rows: the suffix
positions c+1..T of the proposal generated at v+.  Segment 0 of a chain is the
root state, whose rows cover positions root_cut+1..T.

Node arrays use these codes for ``req`` (the request whose proposal the
decision at the node needs): a segment id >= 0, LEAF (-1, not expanded) or
DEFERRED (-2, expanded but its request was deferred; the walk stops there).

Only random draws and bookkeeping live here; no probability is computed.
"""

from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field

import numpy as np

LEAF = -1
DEFERRED = -2


@dataclass
class ChainTree:
    """One chain's prefetched subtree, with node and segment ids local to it."""

    T: int
    # segments: index 0 is the root state
    seg_cut: list = field(default_factory=list)
    seg_src: list = field(default_factory=list)
    # nodes: index 0 is the root v0
    acc: list = field(default_factory=list)
    rej: list = field(default_factory=list)
    req: list = field(default_factory=list)
    parent: list = field(default_factory=list)
    node_cut: list = field(default_factory=list)
    node_state: list = field(default_factory=list)
    depth: list = field(default_factory=list)
    deferred_cut: dict = field(default_factory=dict)

    @classmethod
    def new(cls, T: int) -> "ChainTree":
        t = cls(T=T)
        t.seg_cut.append(T)      # fixed by finalize_root_cut()
        t.seg_src.append(-1)
        t._add_node(parent=-1, cut=T, state=0, depth=0)
        return t

    def _add_node(self, parent, cut, state, depth) -> int:
        self.acc.append(LEAF)
        self.rej.append(LEAF)
        self.req.append(LEAF)
        self.parent.append(parent)
        self.node_cut.append(cut)
        self.node_state.append(state)
        self.depth.append(depth)
        return len(self.acc) - 1

    def expand(self, v: int, c: int) -> tuple[int, int, bool]:
        """Expand node v with a drawn cut c; returns (v+, v-, feasible)."""
        assert self.req[v] == LEAF, "node expanded twice"
        d = self.depth[v] + 1
        a = self._add_node(parent=v, cut=c, state=-1, depth=d)
        b = self._add_node(parent=v, cut=self.node_cut[v],
                           state=self.node_state[v], depth=d)
        self.acc[v] = a
        self.rej[v] = b
        if c <= self.node_cut[v]:                      # Condition 1
            s = len(self.seg_cut)
            self.seg_cut.append(int(c))
            self.seg_src.append(int(self.node_state[v]))
            self.req[v] = s
            self.node_state[a] = s
            return a, b, True
        self.req[v] = DEFERRED
        self.deferred_cut[v] = int(c)
        return a, b, False

    @property
    def n_requests(self) -> int:
        return len(self.seg_cut) - 1

    def suffix_tokens(self) -> int:
        """Sum over feasible requests of T - c_i (the scored proposal tokens)."""
        return int(sum(self.T - c for c in self.seg_cut[1:]))

    def finalize_root_cut(self, root_cut: int | None = None) -> None:
        """Set the root segment to cover the positions the requests need.

        A request i proposing from the state x_{0:c_src} + y^src reads root rows
        for positions c_i+1..c_src, so the root must cover min_i c_i + 1..T.
        """
        if root_cut is None:
            root_cut = min(self.seg_cut[1:], default=self.T)
        self.seg_cut[0] = int(root_cut)


def bfs_tree(rng: np.random.Generator, T: int, n_pf: int,
             depth_cap: int | None = None) -> ChainTree:
    """BFS request collection with deferral (PreSTO section 3.2, step (1)).

    Cuts are drawn from Unif{0..T-1}.  ``depth_cap`` is the K - k cap of
    Appendix C.1: nodes at depth >= depth_cap are not expanded.
    """
    t = ChainTree.new(T)
    queue = deque([0])
    while queue and t.n_requests < n_pf:
        v = queue.popleft()
        if depth_cap is not None and t.depth[v] >= depth_cap:
            continue
        c = int(rng.integers(0, T))
        a, b, ok = t.expand(v, c)
        if ok:
            queue.append(a)
        queue.append(b)
    t.finalize_root_cut()
    return t


def spine_tree(rng: np.random.Generator, T: int, n_pf: int, spine_depth: int,
               p_rej: float) -> ChainTree:
    """A unary-heavy subtree, as a predictive traversal tends to select.

    A spine of up to ``spine_depth`` expanded nodes leaves the root; at each
    spine node the path continues through the rejection child with
    probability p_rej and through the acceptance child otherwise.  The rest of
    the budget is spent greedily on the frontier: every frontier node has a
    pre-drawn cut for its acceptance child, and the node whose pre-drawn cut
    is largest (the shortest suffix, the cheapest and most often accepted
    request, as a predictor on the cut fraction c/T would rank it) is
    expanded next.  Every drawn cut follows the feasible conditional law
    c ~ Unif{0..min(cut(v), T-1)}, so no request is deferred (a predictive
    selection keeps candidate nodes only, Appendix C.1).  No node deeper than
    ``spine_depth`` is expanded.
    """
    t = ChainTree.new(T)

    def draw(v: int) -> int:
        return int(rng.integers(0, min(t.node_cut[v], T - 1) + 1))

    frontier: dict = {}
    v = 0
    for _ in range(min(spine_depth, n_pf)):
        a, b, ok = t.expand(v, draw(v))
        assert ok
        if rng.random() < p_rej:
            side, v = a, b
        else:
            side, v = b, a
        if t.depth[side] < spine_depth:
            frontier[side] = draw(side)
    if t.depth[v] < spine_depth:
        frontier[v] = draw(v)
    while frontier and t.n_requests < n_pf:
        w = max(frontier, key=lambda n: (frontier[n], -n))
        c = frontier.pop(w)
        a, b, ok = t.expand(w, c)
        assert ok
        for n in (a, b):
            if t.depth[n] < spine_depth:
                frontier[n] = draw(n)
    t.finalize_root_cut()
    return t


def example5_tree(T: int, c1: int, c2: int) -> ChainTree:
    """The prefetching tree of Figure 8(b) / Example 5 (Appendix B.3).

    v0 is expanded with request (v1, c1), then v1 with request (v3, c2), c2 <= c1;
    v2 = rejection child of v0, v4 = rejection child of v1.  Node ids follow the
    figure's names: v0..v4 are nodes 0..4.
    """
    assert 0 <= c2 <= c1 <= T - 1
    t = ChainTree.new(T)
    a, b, ok = t.expand(0, c1)
    assert ok and (a, b) == (1, 2)
    a, b, ok = t.expand(1, c2)
    assert ok and (a, b) == (3, 4)
    t.finalize_root_cut()
    return t


@dataclass
class Layout:
    """Flat arrays for a batch of chains (global ids, CSR offsets)."""

    T: int
    n_chains: int
    chain_seg0: np.ndarray   # int32 [n_chains+1]
    seg_row0: np.ndarray     # int64 [n_seg+1]
    seg_cut: np.ndarray      # int32 [n_seg]
    seg_src: np.ndarray      # int32 [n_seg]; chain roots -1, requests: global id
    chain_node0: np.ndarray  # int32 [n_chains+1]
    acc: np.ndarray          # int32 [n_nodes]
    rej: np.ndarray          # int32 [n_nodes]
    req: np.ndarray          # int32 [n_nodes]; global segment id, LEAF or DEFERRED
    trees: list

    @property
    def n_seg(self) -> int:
        return int(self.seg_cut.shape[0])

    @property
    def n_rows(self) -> int:
        return int(self.seg_row0[-1])

    @property
    def n_nodes(self) -> int:
        return int(self.acc.shape[0])

    def is_root(self) -> np.ndarray:
        r = np.zeros(self.n_seg, dtype=bool)
        r[self.chain_seg0[:-1]] = True
        return r

    def suffix_tokens(self) -> int:
        """Sum over all requests of T - c_i."""
        m = ~self.is_root()
        return int(np.sum(self.T - self.seg_cut[m].astype(np.int64)))


def assemble_layout(trees: list[ChainTree]) -> Layout:
    """Concatenate chains into global CSR arrays.

    Segment s covers positions seg_cut[s]+1..T; its rows are
    seg_row0[s] .. seg_row0[s+1]-1 in position order.
    """
    assert trees
    T = trees[0].T
    chain_seg0 = [0]
    chain_node0 = [0]
    seg_cut, seg_src, seg_rows = [], [], []
    acc, rej, req = [], [], []
    for t in trees:
        assert t.T == T
        s0 = chain_seg0[-1]
        n0 = chain_node0[-1]
        for s, (c, src) in enumerate(zip(t.seg_cut, t.seg_src)):
            seg_cut.append(c)
            seg_src.append(-1 if s == 0 else s0 + src)
            seg_rows.append(T - c)
        for v in range(len(t.acc)):
            acc.append(n0 + t.acc[v] if t.acc[v] >= 0 else t.acc[v])
            rej.append(n0 + t.rej[v] if t.rej[v] >= 0 else t.rej[v])
            req.append(s0 + t.req[v] if t.req[v] >= 0 else t.req[v])
        chain_seg0.append(s0 + len(t.seg_cut))
        chain_node0.append(n0 + len(t.acc))
    seg_row0 = np.zeros(len(seg_rows) + 1, dtype=np.int64)
    seg_row0[1:] = np.cumsum(np.asarray(seg_rows, dtype=np.int64))
    return Layout(
        T=T, n_chains=len(trees),
        chain_seg0=np.asarray(chain_seg0, dtype=np.int32),
        seg_row0=seg_row0,
        seg_cut=np.asarray(seg_cut, dtype=np.int32),
        seg_src=np.asarray(seg_src, dtype=np.int32),
        chain_node0=np.asarray(chain_node0, dtype=np.int32),
        acc=np.asarray(acc, dtype=np.int32),
        rej=np.asarray(rej, dtype=np.int32),
        req=np.asarray(req, dtype=np.int32),
        trees=list(trees),
    )


def draw_uniforms(rng: np.random.Generator, n: int) -> np.ndarray:
    """Acceptance uniforms u in (0, 1], one per segment (roots unused)."""
    return 1.0 - rng.random(n)
