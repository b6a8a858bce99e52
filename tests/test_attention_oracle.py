"""Pins for oracle/attention.py, and planted mistakes that must fail them.

The attention oracle is fixed to torch's scaled_dot_product_attention in
double (a library routine), to closed forms (equal value rows, a single key,
zero queries, the first causal row), to scipy's logsumexp, and its tile-by-tile
form to its definition.  Each planted mistake (copies of the module with one
textual change, loaded from a temporary file) must fail at least one pin.
"""
import importlib.util
import inspect
import os

import numpy as np
import pytest

from oracle import attention as att

SRC = inspect.getsourcefile(att)


def _qkv(bh, n_q, n_k, d, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((bh, n_q, d)) * scale, rng.standard_normal((bh, n_k, d)) * scale,
            rng.standard_normal((bh, n_k, d)))


def pin_torch_sdpa(m):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    for causal, offset, n_q, n_k in ((False, 0, 37, 53), (True, 0, 40, 40), (True, 13, 20, 33),
                                     (True, -3, 25, 25)):
        q, k, v = _qkv(3, n_q, n_k, 16, seed=n_q + n_k, scale=2.0)
        got = m.attention(q, k, v, causal=causal, offset=offset)
        mask = None
        if causal:
            mask = torch.ones(n_q, n_k, dtype=torch.bool).tril(diagonal=offset)
        ref = F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k),
                                             torch.from_numpy(v), attn_mask=mask).numpy()
        # A query with no visible key: the formula's NaN here; torch returns
        # zeros for such rows by its own convention, so only rows with a key
        # are compared with it.
        seen = np.ones((n_q,), bool) if not causal else (np.arange(n_q) + offset >= 0)
        assert np.all(np.isnan(got[:, ~seen])) and not np.isnan(got[:, seen]).any()
        assert np.allclose(got[:, seen], ref[:, seen], rtol=1e-12, atol=1e-13), (causal, offset)


def pin_online_equals_definition(m):
    for block in (1, 7, 64):
        for causal, offset in ((False, 0), (True, 0), (True, -5)):
            q, k, v = _qkv(2, 30, 45, 8, seed=block, scale=3.0)
            a = m.attention(q, k, v, causal=causal, offset=offset)
            b = m.attention_online(q, k, v, causal=causal, offset=offset, block_n=block)
            ok = ~np.isnan(a)
            assert np.array_equal(np.isnan(a), np.isnan(b))
            assert np.allclose(a[ok], b[ok], rtol=1e-12, atol=1e-14)


def pin_closed_forms(m):
    rng = np.random.default_rng(3)
    q, k, _ = _qkv(1, 9, 12, 4, seed=4, scale=2.0)
    c = rng.standard_normal(4)
    v = np.broadcast_to(c, (1, 12, 4))
    for fn in (m.attention, m.attention_online):
        assert np.allclose(fn(q, k, v), np.broadcast_to(c, (1, 9, 4)), rtol=1e-14, atol=1e-15)
    q, k, v = _qkv(1, 5, 1, 4, seed=5)                    # one key: every row is v[0]
    assert np.allclose(m.attention(q, k, v), np.broadcast_to(v[0, 0], (1, 5, 4)), rtol=1e-15)
    q, k, v = _qkv(1, 6, 10, 4, seed=6)
    zero = m.attention(np.zeros_like(q), k, v)           # equal scores: the mean of v
    assert np.allclose(zero, np.broadcast_to(v[0].mean(axis=0), (1, 6, 4)), rtol=1e-14)
    causal = m.attention(q, k[:, :6], v[:, :6], causal=True)
    assert np.array_equal(causal[0, 0], v[0, 0])          # query 0 sees key 0 only
    assert np.allclose(causal[0, 2], v[0, :3].T @ _softmax(q[0, 2] @ k[0, :3].T / 2.0))
    empty = m.attention(q, k, v, causal=True, offset=-1)  # query 0 sees nothing
    assert np.all(np.isnan(empty[0, 0])) and np.all(np.isfinite(empty[0, 1:]))
    # No key at all is the same as every key masked: the softmax of only -inf
    # (NaN outputs), whose logsumexp is log 0 = -inf.
    none = np.zeros((1, 0, 4))
    hidden = m.attention(q, k, v, causal=True, offset=-10)
    assert np.all(np.isnan(hidden)) and np.all(np.isneginf(m.logsumexp(q, k, causal=True,
                                                                       offset=-10)))
    for fn in (m.attention, m.attention_online):
        out = fn(q, none, none)
        assert out.shape == (1, 6, 4) and np.all(np.isnan(out))
    assert np.all(np.isneginf(m.logsumexp(q, none)))


def _softmax(z):
    e = np.exp(z - z.max())
    return e / e.sum()


def pin_logsumexp(m):
    special = pytest.importorskip("scipy.special")
    q, k, _ = _qkv(2, 11, 17, 8, seed=8, scale=3.0)
    got = m.logsumexp(q, k, causal=True, offset=2)
    for b in range(2):
        for i in range(11):
            s = q[b, i] @ k[b, : min(17, i + 3)].T / np.sqrt(8)
            assert abs(got[b, i] - special.logsumexp(s)) <= 1e-13 * (1 + abs(got[b, i]))


PINS = [pin_torch_sdpa, pin_online_equals_definition, pin_closed_forms, pin_logsumexp]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_attention_oracle_pin(pin):
    pin(att)


MUTANTS = {
    "no_scale": ("s = scale * (q[b] @ k[b].T)", "s = (q[b] @ k[b].T)"),
    "mask_off_by_one": ("return np.arange(n_k)[None, :] <= np.arange(n_q)[:, None] + offset",
                        "return np.arange(n_k)[None, :] < np.arange(n_q)[:, None] + offset"),
    "no_normalise": ("out[b] = (e @ v[b]) / e.sum(axis=1, keepdims=True)", "out[b] = e @ v[b]"),
    "empty_keys_give_zero": ("out[b] = (e @ v[b]) / e.sum(axis=1, keepdims=True)",
                             "out[b] = (e / e.sum(axis=1, keepdims=True)) @ v[b]"),
    "online_no_rescale": ("acc = acc * alpha[:, None] + p @ vt", "acc = acc + p @ vt"),
    "online_l_no_rescale": ("                l_i = l_i * alpha + l_ij",
                            "                l_i = l_i + l_ij"),
    "transposed_v": ("out[b] = (e @ v[b])", "out[b] = (v[b].T @ e.T).T[:, ::-1]"),
    "lse_no_ref": ("out[b] = ref + np.log(", "out[b] = np.log("),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_attention_planted_mistake_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, name
    path = tmp_path / ("mutant_%s.py" % name)
    path.write_text(src.replace(before, after))
    spec = importlib.util.spec_from_file_location("mutant_" + name, str(path))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    caught = []
    for pin in PINS:
        try:
            pin(mod)
        except pytest.skip.Exception:
            continue
        except Exception:
            caught.append(pin.__name__)
    assert caught, "no pin fails on planted mistake " + name
