"""Incremental decode state, fp64 reference (test infrastructure).

Only the tests may import this module; the product library shares no code
with it.  It restates the serving-side state the pages describe, one token at
a time, on top of the oracle's own steps:

* a growing cache of completed compressed entries (CSA KV, CSA indexer keys,
  HCA KV), each entry stored once its block of m tokens is complete;
* a bounded state per request: the window of the last n_win raw rows and the
  unfinished compression tail (the rows of the current block, plus, in the
  two-branch mode, the previous block's second-branch rows that the next
  entry pools).

["DeepSeek-V4" book, ch.5 "What is retained during decode"; ch.13 "Bounded
state per request": when a token arrives the window advances and the
compression state changes; when a block completes its summary moves into the
growing cache.]

Each arriving token at position t is stored as the prefill path stores it (the
raw row rotated at t and rounded to the storage dtype; a completed block
compressed in fp64, rotated at its last position and rounded once), and the
query at t then reads exactly what a prefill query at t reads, so the outputs
match the prefill oracle step for step.
"""
from __future__ import annotations

import numpy as np

import oracle as orc


class LayerState:
    """One sequence of one compressed layer: KV (and, for CSA, indexer keys)."""

    def __init__(self, s: dict, *, m: int, csa: bool, overlap: int = 0):
        self.s, self.m, self.csa, self.overlap = s, m, csa, overlap
        self.dt, self.r, self.th, self.n_win = s["dtype"], s["rope_dims"], s["theta"], s["n_win"]
        self.t = 0                                   # tokens seen
        self.entries = []                            # stored KV entries (float64, dtype values)
        self.keys = []                               # stored indexer keys (CSA)
        self.win = []                                # (position, stored raw row), oldest first
        self.tail = []                               # this block's rows so far (dict of arrays)
        self.prev = None                             # previous block's rows (two-branch mode)

    # ------------------------------------------------------------ arrival
    def push(self, row: dict, bias: dict) -> None:
        """Token t: row holds its C, Z (and Ck, Zk; second-branch Cb, Zb, Ckb, Zkb
        in the two-branch mode) as 1-D storage arrays; bias the layer's biases."""
        t = self.t
        raw = orc.rope_rows(row["C"][None], t, self.r, self.th, self.dt)[0]
        self.win.append((t, raw))
        if len(self.win) > self.n_win:
            self.win.pop(0)
        self.tail.append(row)
        if len(self.tail) == self.m:
            self._complete(bias)
        self.t += 1

    def _pool(self, key_c: str, key_z: str, bias, key_cb=None, key_zb=None, biasb=None) -> np.ndarray:
        # one entry, unrotated, in fp64: the block's own slots, plus the previous
        # block's second-branch slots in the two-branch mode
        cur_c = np.stack([r[key_c] for r in self.tail])
        cur_z = np.stack([r[key_z] for r in self.tail])
        if not self.overlap:
            return orc.compress(cur_c, cur_z, bias, self.m, rope_dims=0, out_dtype="f64")[0]
        cb = np.stack([r[key_cb] for r in self.tail])
        zb = np.stack([r[key_zb] for r in self.tail])
        if self.prev is None:
            return orc.compress(cur_c, cur_z, bias, self.m, overlap=1, Cb=cb, Zb=zb, biasb=biasb,
                                rope_dims=0, out_dtype="f64")[0]
        pc = np.concatenate([np.stack([r[key_c] for r in self.prev]), cur_c])
        pz = np.concatenate([np.stack([r[key_z] for r in self.prev]), cur_z])
        pcb = np.concatenate([np.stack([r[key_cb] for r in self.prev]), cb])
        pzb = np.concatenate([np.stack([r[key_zb] for r in self.prev]), zb])
        return orc.compress(pc, pz, bias, self.m, overlap=1, Cb=pcb, Zb=pzb, biasb=biasb,
                            rope_dims=0, out_dtype="f64")[1]

    def _complete(self, bias: dict) -> None:
        i = len(self.entries)                        # block index; last position (i+1)m - 1
        e = self._pool("C", "Z", bias["bias"], "Cb", "Zb", bias.get("biasb"))
        e = orc.rope(e, float((i + 1) * self.m - 1), self.r, self.th)
        self.entries.append(orc.round_to(e, self.dt))
        if self.csa:
            k = self._pool("Ck", "Zk", bias["biask"], "Ckb", "Zkb", bias.get("biaskb"))
            self.keys.append(orc.round_to(k, self.dt))
        self.prev = self.tail if self.overlap else None
        self.tail = []

    # ------------------------------------------------------------- state
    def state_rows(self) -> dict:
        """Sizes of the bounded state and of the growing cache."""
        return {"window": len(self.win), "tail": len(self.tail),
                "prev": len(self.prev) if self.prev is not None else 0,
                "entries": len(self.entries)}

    def _cache(self, rows: list) -> np.ndarray:
        c = self.s["c"] if rows is self.entries else self.s.get("dI", self.s["c"])
        if not rows:                                 # no entry yet: one invisible zero row
            return np.zeros((1, c))
        return np.stack(rows)

    # ------------------------------------------------------------- query
    def query(self, q, sink, qI=None, w=None) -> dict:
        """The query at the latest position t: CSA scores -> top-k -> attention
        over the selected entries, the window and the sink; HCA attention over
        every visible entry, the window and the sink."""
        t = self.t - 1
        pos = np.array([t], np.int64)
        p0 = self.win[0][0]
        raw = orc._storage(np.stack([r for _, r in self.win]), self.dt)
        kvc = orc._storage(self._cache(self.entries), self.dt)
        res = {}
        idx = None
        if self.csa:
            kI = orc._storage(self._cache(self.keys), self.dt)
            sc = orc.index_scores(qI[None], w[None], pos, kI, self.m)
            idx, cnt = orc.topk(sc, pos, self.m, self.s["top_k"])
            res.update(scores=sc[0], idx=idx[0], cnt=int(cnt[0]))
        res["out"] = orc.attend(q[None], pos, kvc, self.m, raw, p0, sink, idx=idx,
                                n_win=self.n_win, rope_dims=self.r, theta=self.th,
                                derotate=self.s.get("derotate", 1))[0]
        return res
