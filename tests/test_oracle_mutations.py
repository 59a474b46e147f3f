"""The oracle's pins catch plausible mistakes planted in the oracle.

Each mutant below replaces one function of the float64 oracle (in memory, for one test, through
monkeypatch) by a version with one plausible mistake: a dropped term, a wrong sign, index, base
or denominator, an overwritten accumulation. Then every pin of tests/test_oracle_pins.py runs,
with its own parametrisations. A mutant is caught when at least one pin fails; every mutant must
be caught. The unmutated oracle must pass every pin through the same runner, which shows the
runner itself reports failures only where there are some.

Mistakes are planted in the oracle only, on the CPU; nothing here touches the product path.
"""
import importlib.util
import itertools
import os

import numpy as np
import pytest

import oracle
import oracle.flce_oracle as OM

PINS_FILE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "test_oracle_pins.py")


def _load_pins():
    spec = importlib.util.spec_from_file_location("oracle_pins_under_mutation", PINS_FILE)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _cases(fn):
    """(label, kwargs) for every parametrisation of a pin function."""
    axes = []
    for mark in getattr(fn, "pytestmark", []):
        if mark.name != "parametrize":
            continue
        names = [n.strip() for n in mark.args[0].split(",")]
        values = [v if len(names) > 1 else (v,) for v in mark.args[1]]
        axes.append([dict(zip(names, v)) for v in values])
    for combo in itertools.product(*axes):
        kw = {}
        for part in combo:
            kw.update(part)
        yield f"{fn.__name__}{kw if kw else ''}", kw


def _run_pins():
    """Run every pin; return (failed, passed) lists of labels (skips are in neither)."""
    pins = _load_pins()
    failed, passed = [], []
    for name in sorted(dir(pins)):
        fn = getattr(pins, name)
        if not (name.startswith("test_") and callable(fn)):
            continue
        for label, kw in _cases(fn):
            try:
                with np.errstate(all="ignore"):
                    fn(**kw)
            except pytest.skip.Exception:
                continue
            except Exception:  # an assertion or an error: the pin did not hold
                failed.append(label)
            else:
                passed.append(label)
    return failed, passed


# ---------------------------------------------------------------- the planted mistakes

def _plant(monkeypatch, name, fn):
    monkeypatch.setattr(OM, name, fn)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, fn)


def _lse_without_max(monkeypatch):
    _plant(monkeypatch, "log_sum_exp", lambda z: np.log(np.exp(z).sum(axis=1)))


def _lse_base_two(monkeypatch):
    def lse(z):
        m = z.max(axis=1)
        return m + np.log2(np.exp(z - m[:, None]).sum(axis=1))
    _plant(monkeypatch, "log_sum_exp", lse)


def _lse_max_added_twice(monkeypatch):
    def lse(z):
        m = z.max(axis=1)
        return 2 * m + np.log(np.exp(z - m[:, None]).sum(axis=1))
    _plant(monkeypatch, "log_sum_exp", lse)


def _logits_permuted_hidden(monkeypatch):
    _plant(monkeypatch, "logits", lambda x_rows, weight: x_rows @ weight[:, ::-1].T)


def _logits_missing_last_hidden(monkeypatch):
    _plant(monkeypatch, "logits", lambda x_rows, weight: x_rows[:, :-1] @ weight[:, :-1].T)


def _dz_sign_flipped(monkeypatch):
    orig = OM.dlogits
    _plant(monkeypatch, "dlogits", lambda z, lse, target, g: -orig(z, lse, target, g))


def _dz_without_onehot(monkeypatch):
    def dz(z, lse, target, g):
        p = np.exp(z - lse[:, None])
        g = np.asarray(g, dtype=np.float64)
        return p * (g[:, None] if g.ndim == 1 else g)
    _plant(monkeypatch, "dlogits", dz)


def _dz_onehot_at_neighbour(monkeypatch):
    orig = OM.dlogits
    _plant(monkeypatch, "dlogits",
           lambda z, lse, target, g: orig(z, lse, (target + 1) % z.shape[1], g))


def _dz_scaled_twice(monkeypatch):
    orig = OM.dlogits

    def dz(z, lse, target, g):
        g = np.asarray(g, dtype=np.float64)
        return orig(z, lse, target, g) * (g[:, None] if g.ndim == 1 else g)
    _plant(monkeypatch, "dlogits", dz)


def _target_shifted(monkeypatch):
    orig = OM._check

    def check(x, weight, target):
        x, weight, target = orig(x, weight, target)
        return x, weight, (target + 1) % weight.shape[0]
    monkeypatch.setattr(OM, "_check", check)


def _mean_loss_over_vocab(monkeypatch):
    orig = OM.forward

    def forward(x, weight, target, reduction="mean", chunk=256):
        loss, lse = orig(x, weight, target, reduction, chunk)
        if reduction == "mean":
            loss = loss * np.shape(x)[0] / np.shape(weight)[0]
        return loss, lse
    _plant(monkeypatch, "forward", forward)


def _sum_returns_mean(monkeypatch):
    orig = OM.forward

    def forward(x, weight, target, reduction="mean", chunk=256):
        loss, lse = orig(x, weight, target, reduction, chunk)
        if reduction == "sum":
            loss = loss / np.shape(x)[0]
        return loss, lse
    _plant(monkeypatch, "forward", forward)


def _mean_grad_not_divided(monkeypatch):
    orig = OM.grad_scale

    def grad_scale(grad_loss, reduction, T):
        return orig(grad_loss, "sum" if reduction == "mean" else reduction, T)
    _plant(monkeypatch, "grad_scale", grad_scale)


def _none_grad_first_token_only(monkeypatch):
    orig = OM.grad_scale

    def grad_scale(grad_loss, reduction, T):
        g = orig(grad_loss, reduction, T)
        return np.full(T, g[0]) if reduction == "none" else g
    _plant(monkeypatch, "grad_scale", grad_scale)


def _backward_with(grad_w_update):
    """The oracle's backward with its grad_weight update replaced by grad_w_update(acc, dz, xc)."""
    def backward(x, weight, target, lse, reduction="mean", grad_loss=1.0, chunk=256):
        x, weight, target = OM._check(x, weight, target)
        lse = np.asarray(lse, dtype=np.float64)
        T = x.shape[0]
        g = OM.grad_scale(grad_loss, reduction, T)
        grad_x = np.empty_like(x)
        grad_w = np.zeros_like(weight)
        for t0 in range(0, T, chunk):
            t1 = min(T, t0 + chunk)
            z = OM.logits(x[t0:t1], weight)
            gc = g[t0:t1] if isinstance(g, np.ndarray) else g
            dz = OM.dlogits(z, lse[t0:t1], target[t0:t1], gc)
            grad_x[t0:t1] = dz @ weight
            grad_w = grad_w_update(grad_w, dz, x[t0:t1])
        return grad_x, grad_w
    return backward


def _grad_weight_overwritten(monkeypatch):
    # the last token chunk's term only
    _plant(monkeypatch, "backward", _backward_with(lambda acc, dz, xc: dz.T @ xc))


def _grad_weight_from_wrong_operand(monkeypatch):
    # dz^T . x with the chunk's token rows of x in reverse order (an index mistake)
    _plant(monkeypatch, "backward", _backward_with(lambda acc, dz, xc: acc + dz.T @ xc[::-1]))


def _grad_x_negated(monkeypatch):
    orig = OM.backward

    def backward(*a, **kw):
        gx, gw = orig(*a, **kw)
        return -gx, gw
    _plant(monkeypatch, "backward", backward)


def _gw_rows_with(dz_column):
    """The oracle's grad_weight_rows with its dz columns formed by dz_column(z, lse, onehot, g)."""
    def grad_weight_rows(x, weight, target, lse, vocab_rows, reduction="mean", grad_loss=1.0,
                         chunk=4096):
        x, weight, target = OM._check(x, weight, target)
        lse = np.asarray(lse, dtype=np.float64).reshape(-1)
        rows = np.asarray(vocab_rows, dtype=np.int64).reshape(-1)
        T = x.shape[0]
        g = OM.grad_scale(grad_loss, reduction, T)
        out = np.zeros((rows.size, x.shape[1]))
        for t0 in range(0, T, chunk):
            t1 = min(T, t0 + chunk)
            zc = OM.logits(x[t0:t1], weight[rows])
            onehot = (target[t0:t1, None] == rows[None, :]).astype(np.float64)
            gc = g[t0:t1, None] if isinstance(g, np.ndarray) else g
            out += dz_column(zc, lse[t0:t1, None], onehot, gc).T @ x[t0:t1]
        return out
    return grad_weight_rows


def _gw_rows_sign_flipped(monkeypatch):
    _plant(monkeypatch, "grad_weight_rows",
           _gw_rows_with(lambda z, lse, oh, g: -(np.exp(z - lse) - oh) * g))


def _gw_rows_without_onehot(monkeypatch):
    _plant(monkeypatch, "grad_weight_rows", _gw_rows_with(lambda z, lse, oh, g: np.exp(z - lse) * g))


def _gw_rows_onehot_at_neighbour(monkeypatch):
    _plant(monkeypatch, "grad_weight_rows",
           _gw_rows_with(lambda z, lse, oh, g: (np.exp(z - lse) - np.roll(oh, 1, axis=1)) * g))


def _gw_rows_without_upstream_gradient(monkeypatch):
    _plant(monkeypatch, "grad_weight_rows", _gw_rows_with(lambda z, lse, oh, g: np.exp(z - lse) - oh))


def _gw_rows_without_lse(monkeypatch):
    _plant(monkeypatch, "grad_weight_rows", _gw_rows_with(lambda z, lse, oh, g: (np.exp(z) - oh) * g))


MUTANTS = {
    "log-sum-exp without the row maximum": _lse_without_max,
    "log-sum-exp in base 2": _lse_base_two,
    "log-sum-exp adds the row maximum twice": _lse_max_added_twice,
    "logits over a permuted hidden axis": _logits_permuted_hidden,
    "logits missing the last hidden term": _logits_missing_last_hidden,
    "dz with its sign flipped": _dz_sign_flipped,
    "dz without the one-hot term": _dz_without_onehot,
    "dz one-hot at the neighbouring vocab id": _dz_onehot_at_neighbour,
    "dz scaled by the upstream gradient twice": _dz_scaled_twice,
    "every target shifted by one": _target_shifted,
    "mean loss divided by V instead of T": _mean_loss_over_vocab,
    "sum reduction returns the mean": _sum_returns_mean,
    "mean gradient not divided by T": _mean_grad_not_divided,
    "none: first token's upstream gradient for all": _none_grad_first_token_only,
    "grad_weight overwritten per token chunk": _grad_weight_overwritten,
    "grad_x negated": _grad_x_negated,
    "grad_weight from token-reversed x": _grad_weight_from_wrong_operand,
    "sampled grad_weight rows with the dz sign flipped": _gw_rows_sign_flipped,
    "sampled grad_weight rows without the one-hot term": _gw_rows_without_onehot,
    "sampled grad_weight rows with the one-hot at the neighbouring row": _gw_rows_onehot_at_neighbour,
    "sampled grad_weight rows without the upstream gradient": _gw_rows_without_upstream_gradient,
    "sampled grad_weight rows without the lse": _gw_rows_without_lse,
}


def test_unmutated_oracle_passes_every_pin_through_the_runner():
    failed, passed = _run_pins()
    assert not failed, failed
    assert len(passed) >= 35  # every pin and its parametrisations ran


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    MUTANTS[name](monkeypatch)
    failed, passed = _run_pins()
    assert failed, f"no pin caught the planted mistake: {name}"
