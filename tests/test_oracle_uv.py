"""Pins of the oracle's W_UV up-projection (drafter-attention page, `DraftDcp`
and `latent_major`: each head's merged 512-dim latent row times that head's
W_UV [512, 128]), and planted mistakes the pins must each catch."""
import numpy as np
import pytest

import oracle.uv as uv


def _brute(out, w):
    T, H, C = len(out), len(out[0]), len(out[0][0])
    J = len(w[0][0])
    y = [[[0.0] * J for _ in range(H)] for _ in range(T)]
    for t in range(T):
        for h in range(H):
            for j in range(J):
                acc = 0.0
                for c in range(C):
                    acc += out[t][h][c] * w[h][c][j]
                y[t][h][j] = acc
    return np.array(y)


def pin_brute_force(f):
    rng = np.random.default_rng(0)
    out = rng.normal(size=(3, 2, 512))
    w = rng.normal(size=(2, 512, 128))
    return np.allclose(f(out, w), _brute(out.tolist(), w.tolist()), rtol=1e-12, atol=1e-12)


def pin_shifted_identity(f):
    # W[h, c, j] = 1 where c == j + 64 h: y[t, h, :] = out[t, h, 64h : 64h + 128]
    T, H = 4, 3
    out = np.arange(T * H * 512, dtype=np.float64).reshape(T, H, 512)
    w = np.zeros((H, 512, 128))
    for h in range(H):
        w[h, np.arange(128) + 64 * h, np.arange(128)] = 1.0
    y = f(out, w)
    return all(np.array_equal(y[:, h, :], out[:, h, 64 * h: 64 * h + 128]) for h in range(H))


def pin_per_head_scale(f):
    # W[h] = (h + 1) on the first 128 latent rows: every output of head h is
    # (h + 1) times the sum of that head's first 128 latent values
    T, H = 2, 4
    out = np.random.default_rng(1).normal(size=(T, H, 512))
    w = np.zeros((H, 512, 128))
    for h in range(H):
        w[h, :128, :] = h + 1
    y = f(out, w)
    return all(np.allclose(y[:, h, :], (h + 1) * out[:, h, :128].sum(-1)[:, None])
               for h in range(H))


PINS = [pin_brute_force, pin_shifted_identity, pin_per_head_scale]


@pytest.mark.parametrize("pin", PINS)
def test_oracle_passes(pin):
    assert pin(uv.uv_project)


def _wrong_head(out, w):
    H = w.shape[0]
    return np.stack([out[:, h, :] @ w[(h + 1) % H] for h in range(H)], axis=1)


def _reshaped_not_transposed(out, w):
    # the latent-contiguous [H, 128, 512] storage read back with a reshape
    wt = np.ascontiguousarray(w.transpose(0, 2, 1)).reshape(w.shape)
    return uv.uv_project(out, wt)


def _dropped_block(out, w):
    o = np.array(out, dtype=np.float64)
    o[:, :, 448:] = 0.0
    return uv.uv_project(o, w)


@pytest.mark.parametrize("mutant", [_wrong_head, _reshaped_not_transposed, _dropped_block])
def test_pins_catch_mutant(mutant):
    caught = [p.__name__ for p in PINS if not p(mutant)]
    assert caught, f"{mutant.__name__} passes every pin"


def test_shape_checks():
    with pytest.raises(AssertionError):
        uv.uv_project(np.zeros((1, 2, 512)), np.zeros((3, 512, 128)))
