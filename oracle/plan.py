"""Verify preprocess: the verification plan of one request (oracle; test infrastructure only).

[TSD-V4] §4.1: before target verification the candidate tree is turned into a verification plan
that says which candidate chains exist and where their compression boundaries fall.  [TSD-V4]
§3.1: each candidate attends to the accepted context and to the ancestors on its own branch only.

Tree convention ([TSD-V4] §5.1 names ``s4_k1_d5`` a 4-step chain verified with budget 5, so the
budget D counts the root): node 0 is the root, the last accepted token, whose K/V are produced in
this pass; ``parents[0] == -1`` and ``0 <= parents[v] < v`` for every other node (topological
numbering).  Node v sits at depth ``depth[v]`` (root 0) and sequence position
``pos[v] = L + depth[v]``, where ``L`` is the request's committed length.

Per node the plan holds
* ``anc[v]``   bitmask of v's ancestors including v itself (bit u set iff u is on root->v);
* ``raw_lo[v]`` the lowest raw position visible from v: ``max(0, pos - W)`` in window mode,
  ``m_min * floor(pos / m_min)`` in remainder mode (only the unfinished block stays raw);
* ``completes[m][v]`` True iff v's token closes a block of compressor m: ``(pos + 1) % m == 0``;
* ``scr_vis[m][v]`` bitmask of v's PROPER ancestors that close a block of m: the scratch-pad
  entries that v may see (a token never sees an entry that contains itself).
"""

from dataclasses import dataclass, field


@dataclass
class Plan:
    anc: list
    depth: list
    pos: list
    raw_lo: list
    completes: dict = field(default_factory=dict)
    scr_vis: dict = field(default_factory=dict)


def validate_parents(parents):
    D = len(parents)
    if D < 1:
        raise ValueError("empty tree")
    if int(parents[0]) != -1:
        raise ValueError("parents[0] must be -1 (the root)")
    for v in range(1, D):
        p = int(parents[v])
        if not (0 <= p < v):
            raise ValueError(f"parents[{v}] = {p} is not a node numbered before {v}")


def build_plan(parents, L, W, tail_mode, ms):
    """The verification plan of one request.

    parents: D ints; L: committed length; W: raw window (tail_mode "window");
    tail_mode: "window" or "remainder"; ms: active compressor block sizes, e.g. (4, 128).
    """
    validate_parents(parents)
    D = len(parents)
    anc, depth = [], []
    for v in range(D):
        mask, dep, u = 0, 0, v
        while True:
            mask |= 1 << u
            if u == 0:
                break
            u = int(parents[u])
            dep += 1
        anc.append(mask)
        depth.append(dep)
    pos = [L + depth[v] for v in range(D)]
    if tail_mode == "window":
        raw_lo = [max(0, pos[v] - W) for v in range(D)]
    elif tail_mode == "remainder":
        m_min = min(ms)
        raw_lo = [m_min * (pos[v] // m_min) for v in range(D)]
    else:
        raise ValueError(f"unknown tail mode {tail_mode!r}")
    completes, scr_vis = {}, {}
    for m in ms:
        completes[m] = [(pos[v] + 1) % m == 0 for v in range(D)]
        vis = []
        for v in range(D):
            bits = 0
            for u in range(D):
                if u != v and (anc[v] >> u) & 1 and completes[m][u]:
                    bits |= 1 << u
            vis.append(bits)
        scr_vis[m] = vis
    return Plan(anc=anc, depth=depth, pos=pos, raw_lo=raw_lo, completes=completes, scr_vis=scr_vis)
