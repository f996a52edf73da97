"""W_UV up-projection of the attention's latent output, in float64.

Test infrastructure only (see the package docstring).

After the heads' partial rows are merged, each (token, head) row of the
512-dim latent output is multiplied by that head's W_UV [512, 128], giving the
head's 128-dim value in the attention output (drafter-attention page,
``DraftDcp``: the head owner merges its heads over the sources and applies
W_UV as a BF16 MMA with FP32 accumulation; ``latent_major``: W_UV is
[H, 512, 128]). The pages round the merged row to BF16 once before the
product and the product to BF16; this definition is the exact product, and
the CUDA path is checked against it at a tolerance derived from those
roundings.
"""
from __future__ import annotations

import numpy as np

D_V = 512
D_OUT = 128


def uv_project(out, w_uv):
    """out: [T, H, 512] latent rows (token-major, then head); w_uv: [H, 512, 128].
    Returns y [T, H, 128] with y[t, h, j] = sum_c out[t, h, c] * w_uv[h, c, j]."""
    o = np.asarray(out, dtype=np.float64)
    w = np.asarray(w_uv, dtype=np.float64)
    T, H, C = o.shape
    assert C == D_V and w.shape == (H, D_V, D_OUT)
    y = np.empty((T, H, D_OUT))
    for h in range(H):
        y[:, h, :] = o[:, h, :] @ w[h]
    return y
