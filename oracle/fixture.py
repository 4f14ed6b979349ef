"""The [Ch37] fixture: 1 layer, B = 1, D = 4, H = 2, d_h = 2, C = 4, f64.

[Ch37] "Predict the third result before running the example" and "Advance
the layer cache one position at a time" print, for three single-row calls from
an empty cache, every rotated key, unrotated value, newest-query weight and
merged output -- but not the layer's weights nor its input rows.  The printed
trace is reproduced at the attention level by these per-head projected rows
(q = k = v per head, unrotated, position p = 0, 1, 2):

  head 0: (cos p, -sin p)      -> rotated key (1, 0) at every p
  head 1: (1, 0), (0, 1), (1, 1)

and the output projection that swaps the two head blocks, y = [o_1, o_0]
(the merge-then-project step of [Ch37] "Bind the state, calculate completely,
then commit").  These rows are a reading (the unpublished weights and inputs
could differ while giving the same projections); the printed numbers are the
pins.

The other reading draws Wq, Wk, Wv, Wo ~ N(0, 1/D) and inputs ~ N(0, 1); it is
pinned only by incremental == full-prefix.
"""

import numpy as np

D, H, DH, C = 4, 2, 2, 4
ROPE_BASE = 10000.0


def head_swap_projection():
    """Wo for y = merged @ Wo that maps [o_0, o_1] to [o_1, o_0]."""
    Wo = np.zeros((D, D))
    Wo[0, 2] = Wo[1, 3] = Wo[2, 0] = Wo[3, 1] = 1.0
    return Wo


def split_heads(x):
    """[B, D] -> [B, H, d_h] (head h takes features h*d_h .. h*d_h + d_h - 1)."""
    return x.reshape(x.shape[0], H, DH)


def merge_heads(o):
    """[B, H, d_h] -> [B, D]."""
    return o.reshape(o.shape[0], H * DH)
