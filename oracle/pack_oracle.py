"""Oracle of the packed exchange layout -- test infrastructure only (imported
by tests/, __graft_entry__.smoke() and bench.py's CPU legs, never by the
library).

"DMuon" summary, section 2.1: gradients are reduced into owner-contiguous
buffers before the orthogonalisation and the updated parameters are
published from them afterwards; section 2.3: every matrix has one owner.
The layout, restated plainly: rank r's segment holds the matrices it owns in
ascending index, each starting at the next multiple of `align` within the
segment; every segment is as long as the longest one rounded up to `align`;
segment r starts at r times that length.  `pack` copies each matrix's
row-major elements to its offset; nothing else in the buffer is written.
"""
import numpy as np


def layout(shapes, owners, ranks, align):
    """(offset per matrix, segment length), both in elements."""
    local = [0] * len(shapes)
    ends = [0] * ranks
    for i, (m, n) in enumerate(shapes):
        r = owners[i]
        start = -(-ends[r] // align) * align          # round up to a multiple of align
        local[i] = start
        ends[r] = start + m * n
    seg = max([-(-e // align) * align for e in ends] + [0])
    return [owners[i] * seg + local[i] for i in range(len(shapes))], seg


def pack(mats, offsets, total, fill=0):
    """The packed buffer of `total` elements (numpy), `fill` between matrices."""
    out = np.full(total, fill, dtype=mats[0].dtype if mats else np.float32)
    for a, off in zip(mats, offsets):
        flat = np.ascontiguousarray(a).reshape(-1)
        out[off:off + flat.size] = flat
    return out
