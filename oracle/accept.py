"""Accepted-path selection: the greedy acceptance walk (oracle; test infrastructure only).

[TSD-V4] §3.2 and §4.1: after verification the system picks one specific root-to-node path through
the tree and keeps only its results.  Greedy verification: the target model's token at node u is
``target[u]`` (the token it predicts after the sequence prefix + path(u)); a child c of u is
accepted when its draft token equals ``target[u]``.

Walk: start at the root (always accepted, it is the last accepted token); repeatedly move to the
lowest-numbered child whose draft token equals the target token of the current node; stop when no
child matches.  The accepted length counts the root, and the bonus token is the target token of the
last accepted node (the token the next round starts from).
"""


def accept_walk(parents, draft, target):
    """Returns (accept_len, path, bonus) for one request."""
    D = len(parents)
    cur = 0
    path = [0]
    while True:
        nxt = None
        for c in range(1, D):
            if int(parents[c]) == cur and int(draft[c]) == int(target[cur]):
                nxt = c
                break
        if nxt is None:
            break
        path.append(nxt)
        cur = nxt
    return len(path), path, int(target[cur])
