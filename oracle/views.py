"""Matrix views: how one stored 2-D weight splits into independent matrices.

Follows "build_parameter_groups" (kimi-k3 docs), sections "Recording
independent matrix geometry" and "The layout declarations are literal, not
conceptual reshapes", and the fused-matrix splitting section of
"Qwen3.8-Flash-Next notes / Optimizer" (section 4, split -> orthogonalize
each -> gather back).

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""


class ViewError(ValueError):
    """Raised for a view that the view-registration rules refuse."""


def validate_view(rows, cols, view=None, split=None):
    """Check a view against the registration rules and return it normalised.

    Rules (build_parameter_groups, "Recording independent matrix geometry"):
    every shape entry is a positive integer, and flattening the view's
    leading axes gives back the stored two-dimensional weight shape.  The
    last view axis is the stored column count; the product of all other axes
    is the stored row count.

    Reading for the split sizes (the page's W_UKV example, view (2, 10, 8)
    with split (4, 6) separating K from V inside each head): they partition
    the second-to-last (row) axis of every leading index, so they must be
    positive and sum to that axis.

    Returns ``(view, split)`` as tuples; a missing view is the plain
    ``(rows, cols)`` matrix and a missing split is the whole row axis.
    """
    if not (isinstance(rows, int) and isinstance(cols, int)) or rows <= 0 or cols <= 0:
        raise ViewError("stored shape must be positive integers")
    if view is None:
        view = (rows, cols)
    view = tuple(view)
    if len(view) < 2:
        raise ViewError("a view has at least a row axis and a column axis")
    for s in view:
        if not isinstance(s, int) or s <= 0:
            raise ViewError("every view entry must be a positive integer")
    lead = 1
    for s in view[:-1]:
        lead *= s
    if lead != rows or view[-1] != cols:
        raise ViewError("flattened leading view axes must equal the stored shape")
    r = view[-2]
    if split is None:
        split = (r,)
    split = tuple(split)
    if len(split) == 0 or any((not isinstance(s, int)) or s <= 0 for s in split):
        raise ViewError("split sizes must be positive integers")
    if sum(split) != r:
        raise ViewError("split sizes must sum to the view's row axis")
    return view, split


def sub_matrices(rows, cols, view=None, split=None):
    """List the independent matrices of a stored weight.

    Each entry is ``(row_start, m, n)``: rows ``[row_start, row_start + m)`` of
    the stored row-major ``rows x cols`` weight, all ``n = cols`` columns.

    The leading axes of the view enumerate blocks of ``r`` consecutive stored
    rows (the page's (32, 8) weight viewed as (2, 16, 8) is two (16, 8)
    matrices; (24, 8) viewed as (3, 2, 4, 8) is six (4, 8) matrices).  Inside
    each block the split sizes cut consecutive row ranges (the page's (20, 8)
    weight viewed as (2, 10, 8) with split (4, 6) is, per head, a 4-row K
    matrix followed by a 6-row V matrix).
    """
    view, split = validate_view(rows, cols, view, split)
    r = view[-2]
    n_blocks = rows // r
    out = []
    for b in range(n_blocks):
        start = b * r
        for s in split:
            out.append((start, s, cols))
            start += s
    return out
