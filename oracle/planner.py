"""Owner planner, as longest-processing-time (LPT) greedy.

Oracle module: test infrastructure only.

"Riassunto Tecnico: MatrixFSDP" §Metodologia 2, "Metadati MatrixShard & Global
Planner": a global planner assigns each 2D matrix one owner rank so that the
resident bytes and the optimizer work are balanced across ranks.  The pages do
not give the algorithm.  Reading taken:

    bytes_i = rows_i * cols_i * 2                      (bf16 residency)
    flops_i = k * (4 m^2 n + 2 m^3), m = min, n = max  (NS work)
    cost_i  = w_bytes * bytes_i / sum(bytes) + w_flops * flops_i / sum(flops)

Matrices are taken in order of decreasing cost (ties by increasing index) and
each goes to the rank with the smallest accumulated cost (ties by smallest
rank).  Sums run in index order in float64 so that any implementation doing
the same IEEE operations in the same order reproduces the plan bit for bit.
"""


def matrix_bytes(rows, cols):
    return float(rows) * float(cols) * 2.0


def matrix_flops(rows, cols, steps):
    m, n = (rows, cols) if rows <= cols else (cols, rows)
    m = float(m)
    n = float(n)
    return float(steps) * (4.0 * m * m * n + 2.0 * m * m * m)


def costs(shapes, steps, w_bytes=1.0, w_flops=1.0):
    b = [matrix_bytes(r, c) for r, c in shapes]
    f = [matrix_flops(r, c, steps) for r, c in shapes]
    sb = 0.0
    for x in b:
        sb += x
    sf = 0.0
    for x in f:
        sf += x
    out = []
    for bi, fi in zip(b, f):
        cb = bi / sb if sb > 0 else 0.0
        cf = fi / sf if sf > 0 else 0.0
        out.append(w_bytes * cb + w_flops * cf)
    return out


def plan_owners(shapes, world, steps, w_bytes=1.0, w_flops=1.0):
    """Return (owner list, per-rank load list)."""
    if world <= 0:
        raise ValueError("world must be positive")
    cost = costs(shapes, steps, w_bytes, w_flops)
    order = sorted(range(len(shapes)), key=lambda i: (-cost[i], i))
    load = [0.0] * world
    owner = [-1] * len(shapes)
    for i in order:
        best = 0
        for r in range(1, world):
            if load[r] < load[best]:
                best = r
        owner[i] = best
        load[best] += cost[i]
    return owner, load
