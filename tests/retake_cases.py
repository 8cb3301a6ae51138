"""Constructed score rows for the retake parity cases (test input only).

A block whose sum of p exceeds 2^32 moves the running reference to its max
and is taken again ("Learn: The Memory Wall & FlashAttention", section 8,
conditional rescaling: the kernel's bound is on the block's sum).  These rows
put that retake where what O already holds keeps a visible share of the
weight.
"""
import numpy as np
import torch

SUM_LIMIT = 2.0 ** 32
LOG2E = 1.4426950408889634


def retake_scores(head, N=512):
    """Scores (natural log units, scale 1) of every row for head `head`:
    uniform in [0, 1) but for key block 2 (keys 256-383):
      0: its last 32 keys at 19 and key 296 at 24.  The last keys alone pass
         the 2^32 bound on a block's sum of p; the whole block does not, so
         the reference moves by about 33 (base 2) after those keys were
         weighed, and they keep about 18 % of the block's weight;
      1: its last 32 keys at 24 (they alone fail the bound);
      2: keys 296 and 356 at 12 (a rise of about 17: no retake).
    The values are bf16-exact."""
    g = torch.Generator().manual_seed(900 + head)
    s = torch.rand(N, generator=g)
    if head == 0:
        s[352:384] = 19.0
        s[296] = 24.0
    elif head == 1:
        s[352:384] = 24.0
    else:
        s[296] = 12.0
        s[356] = 12.0
    return s.to(torch.bfloat16)


def reference_path(s, tail_first=True):
    """The kernel's rule for the running reference, on one row of scores s
    (natural units, scale 1), per 128-key block: the first block sets m from
    its max; a block whose sum of p = 2^(s log2 e - m) exceeds 2^32 moves m to
    its max.  With tail_first (the d = 64 kernel) a block's last 32 keys are
    tested on their own first.  Returns (block, event, share of the block's
    weight the last 32 keys keep after the move) per retake."""
    x_all = np.asarray(s, dtype=np.float64) * LOG2E
    m, events = -np.inf, []
    for j in range(len(x_all) // 128):
        x = x_all[128 * j:128 * j + 128]
        if m == -np.inf:
            m = x.max()
        if tail_first and np.exp2(x[96:] - m).sum() > SUM_LIMIT:
            m = max(m, x.max())
            events.append((j, "tail", None))
        if np.exp2(x - m).sum() > SUM_LIMIT:
            m = max(m, x.max())
            w = np.exp2(x - m)
            events.append((j, "block", float(w[96:].sum() / w.sum())))
    return events
