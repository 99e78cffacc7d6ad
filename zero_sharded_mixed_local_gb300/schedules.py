"""Host-side helpers around the step: the learning-rate schedule and the
per-layer learning-rate groups of spectral muP.

Nothing here touches the GPU; the results feed zero1_step (lr) and
zero1_plan_create_grouped (groups and scales).
"""
import math

import numpy as np

from .binding import MAX_GROUPS

HIDDEN, NORM, EMBEDDING = 0, 1, 2


def lr_at(step, lr, warmup_steps, decay_steps, min_lr, decay_style="cosine"):
    """Learning rate at 1-based ``step``.

    The Nanotron guide's config sets learning_rate, lr_warmup_steps,
    lr_decay_steps and min_decay_lr without naming the curves.  Reading
    taken: a linear warm-up from lr/warmup_steps to lr over the first
    warmup_steps steps, then a decay from lr to min_lr over the next
    decay_steps steps ("cosine": half a cosine wave; "linear": a straight
    line; "constant": no decay), then min_lr.
    """
    if step < 1:
        raise ValueError("steps count from 1")
    if decay_style not in ("cosine", "linear", "constant"):
        raise ValueError("unknown decay_style %r" % decay_style)
    if warmup_steps > 0 and step <= warmup_steps:
        return lr * step / warmup_steps
    k = step - warmup_steps
    if decay_style == "constant" or decay_steps <= 0:
        return lr
    if k >= decay_steps:
        return min_lr
    frac = k / decay_steps
    if decay_style == "linear":
        return min_lr + (lr - min_lr) * (1.0 - frac)
    return min_lr + (lr - min_lr) * 0.5 * (1.0 + math.cos(math.pi * frac))  # cosine


def param_kind(name):
    """'norm', 'embedding' (input embedding or output head) or 'hidden' from a parameter name."""
    n = name.lower()
    if "norm" in n:
        return "norm"
    if "embed" in n or "lm_head" in n or "wte" in n:
        return "embedding"
    return "hidden"


def mup_groups(names, d_model, base_d_model=1.0, weight_decay_norms=False):
    """Parameter groups for spectral muP ("Nanotron Guide", "3. Spectral muTransfer":
    eta_hidden = eta_0 / d_model).

    Hidden weight matrices go to group 0 with an lr multiplier of
    base_d_model / d_model (base_d_model = 1 is the page's formula as printed;
    set it to the width the base lr was tuned at to transfer that lr), norm
    weights to group 1 (no weight decay unless asked), embeddings and the
    output head to group 2 (base lr).  Returns (groups, lr_scale, wd_scale)
    for Plan(..., groups=, lr_scale=, wd_scale=).
    """
    kinds = [param_kind(n) for n in names]
    groups = np.array([{"hidden": HIDDEN, "norm": NORM, "embedding": EMBEDDING}[k] for k in kinds], np.uint8)
    lr_scale = np.ones(MAX_GROUPS)
    wd_scale = np.ones(MAX_GROUPS)
    lr_scale[HIDDEN] = float(base_d_model) / float(d_model)
    wd_scale[NORM] = 1.0 if weight_decay_norms else 0.0
    return groups, lr_scale, wd_scale
