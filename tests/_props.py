"""Property checks that characterise the routing-control steps declaratively.

They restate what each step must satisfy, not how the oracle computes it, so
that a slip in the oracle's procedure (a wrong index, a dropped condition, a
wrong tie-break) fails them.  Used on tiny random inputs and on the synthetic
workloads.
"""
from __future__ import annotations

import numpy as np


def sere_expected(ids0, g0, k, kp, rho, sim, protect):
    """For every token, the expert -> gate mapping and the slot position each
    expert must end in, from the rules of SERE (sec. 4.1 / 4.2 of the SERE
    article): candidates are the batch union P of primaries; a non-protected
    secondary outside P goes to its most similar member of P (lower id on
    ties) when that similarity strictly exceeds rho; gates of slots that land
    on the same expert add up."""
    T = ids0.shape[0]
    rho32 = np.float32(rho)
    P = sorted(set(int(v) for v in ids0[:, :kp].ravel()))
    out = []
    for t in range(T):
        target = []
        for r in range(k):
            s = int(ids0[t, r])
            if r < kp or s in P or (protect is not None and protect[s]):
                target.append(s)
                continue
            best = min(P, key=lambda p: (-float(sim[s, p]), p))
            target.append(best if np.float32(sim[s, best]) > rho32 else s)
        gates = {}
        for r in range(k):
            gates.setdefault(target[r], []).append((r, np.float32(g0[t, r])))
        pos = {}
        orig = [int(v) for v in ids0[t, :k]]
        for e in gates:
            pos[e] = orig.index(e) if e in orig else min(r for r in range(k) if target[r] == e)
        out.append((gates, pos))
    return P, out


def check_sere(ids0, g0, ids1, g1, k, kp, rho, sim, protect, stats=None):
    P, exp = sere_expected(ids0, g0, k, kp, rho, sim, protect)
    for t, (gates, pos) in enumerate(exp):
        filled = set()
        for e, parts in gates.items():
            q = pos[e]
            assert ids1[t, q] == e, (t, q, ids1[t], e)
            total = sum(float(v) for _, v in parts)
            assert abs(float(g1[t, q]) - total) <= 1e-6 * max(1.0, abs(total)), (t, e, g1[t, q], total)
            # the holder's gate plus the merged ones in rank order, each an fp32 add
            holder = [v for r, v in parts if r == q]
            rest = [v for r, v in parts if r != q]
            acc = holder[0] if holder else np.float32(0)
            for v in rest:
                acc = np.float32(acc + v)
            if holder:
                assert g1[t, q] == acc, (t, e, g1[t, q], acc)
            filled.add(q)
        for q in range(k):
            if q not in filled:
                assert ids1[t, q] == -1 and g1[t, q] == 0.0, (t, q, ids1[t], g1[t])
    before = set(int(v) for v in ids0[:, :k].ravel())
    after = set(int(v) for v in ids1[:, :k].ravel() if v >= 0)
    assert after <= before
    assert set(P) <= after
    if stats is not None:
        assert stats[0] == len(before) and stats[1] == len(P) and stats[2] == len(after)
    return P


def capacity_check(ids, gates, token_w, k, R, gamma, N, out_ids, out_gates, status, load, C, fixed):
    """Verify a capacity dispatch against its rules without re-running it:
    phase 1 admits, per expert, exactly the pairs whose higher-or-equal
    priority cumulative weight (gate desc, token asc) stays within C; in each
    overflow round every token with a pending slot proposes its lowest-rank
    pending slot to its rank-(k+i) expert, and each expert admits exactly the
    proposals whose cumulative weight on top of its load stays within C."""
    T = ids.shape[0]
    Ce = (lambda e: int(C[e])) if np.ndim(C) > 0 else (lambda e: int(C))   # per-expert or static capacity
    wq = [fixed(float(token_w[t]) if token_w is not None else 1.0) for t in range(T)]
    # phase 1
    load_ref = np.zeros(N, dtype=np.int64)
    pending = {t: [] for t in range(T)}
    for e in range(N):
        pairs = [(t, r) for t in range(T) for r in range(k) if ids[t, r] == e]
        pairs.sort(key=lambda p: (-float(gates[p[0], p[1]]), p[0]))
        for j, (t, r) in enumerate(pairs):
            need = sum(wq[tt] for tt, _ in pairs[: j + 1])
            if need <= Ce(e):
                assert status[t, r] == 0 and out_ids[t, r] == e, ("phase1 admit", t, r)
                load_ref[e] += wq[t]
            else:
                assert status[t, r] != 0, ("phase1 overflow", t, r)
                pending[t].append(r)
    # overflow rounds
    for i in range(R - k):
        props = {}
        for t in range(T):
            if pending[t]:
                r = min(pending[t])
                props.setdefault(int(ids[t, k + i]), []).append((t, r))
        for e, lst in props.items():
            lst.sort(key=lambda p: (-float(gates[p[0], p[1]]), p[0]))
            base = load_ref[e]
            adm = 0
            for j, (t, r) in enumerate(lst):
                need = base + sum(wq[tt] for tt, _ in lst[: j + 1])
                if need <= Ce(e):
                    assert status[t, r] == 1 and out_ids[t, r] == e, ("round admit", i, t, r)
                    adm += wq[t]
                    pending[t].remove(r)
            load_ref[e] += adm
    for t in range(T):
        for r in pending[t]:
            assert status[t, r] == 2 and out_ids[t, r] == -1 and out_gates[t, r] == 0.0, ("drop", t, r)
    for t in range(T):
        for r in range(k):
            if status[t, r] != 2:
                assert out_gates[t, r] == gates[t, r]
    assert np.array_equal(load_ref, load)
    assert (load <= C).all()
    return load_ref
