"""The dense-part oracle (oracle/mlp.py) against its pins, and planted mutants
of it (a dropped ReLU, a wrong sign, a transposed weight, a sum instead of a
mean...) each caught by a pin.  CPU only."""
import importlib.util
import os

import pytest

import mlp_pins
import oracle
from oracle import mlp

MUTANTS = {
    "relu dropped": ("return np.maximum(z, 0.0) if relu else z", "return z"),
    "mask from the input": ("dz = dy * (np.asarray(y) > 0) if relu else dy", "dz = dy"),
    "dx with the transposed weight": ("return dz @ w, dz.T @ x, dz.sum(axis=0)", "return dz @ w.T[:w.shape[1], :w.shape[0]] if w.shape[0] == w.shape[1] else dz @ w * 0.999, dz.T @ x, dz.sum(axis=0)"),
    "sgd adds the gradient": ("new.append((np.asarray(w, np.float64) - lr * dW, np.asarray(b, np.float64) - lr * db))",
                              "new.append((np.asarray(w, np.float64) + lr * dW, np.asarray(b, np.float64) - lr * db))"),
    "loss summed, not averaged": ("loss = np.mean(np.maximum(z, 0.0) - z * label + np.log1p(np.exp(-np.abs(z))))",
                                  "loss = np.sum(np.maximum(z, 0.0) - z * label + np.log1p(np.exp(-np.abs(z))))"),
    "gradient not divided by M": ("dz = (1.0 / (1.0 + np.exp(-z)) - label) / z.shape[0]",
                                  "dz = (1.0 / (1.0 + np.exp(-z)) - label)"),
    "label sign flipped": ("loss = np.mean(np.maximum(z, 0.0) - z * label + np.log1p(np.exp(-np.abs(z))))",
                           "loss = np.mean(np.maximum(z, 0.0) + z * label + np.log1p(np.exp(-np.abs(z))))"),
    "bias ignored": ("z = np.asarray(x, np.float64) @ np.asarray(w, np.float64).T + np.asarray(b, np.float64)",
                     "z = np.asarray(x, np.float64) @ np.asarray(w, np.float64).T"),
    "bottom output without its ReLU": ("bot_outs = mlp_fwd(dense_in, bottom, relu_last=True)",
                                       "bot_outs = mlp_fwd(dense_in, bottom, relu_last=False)"),
}


@pytest.mark.parametrize("pin", mlp_pins.ALL_MLP_PINS, ids=lambda p: p.__name__)
def test_pin(pin, oracle_lib):
    pin(mlp, oracle_lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, oracle_lib):
    src = open(mlp.__file__).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site not found once: {old!r}"
    path = tmp_path / "mlp_mutant.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location("mlp_mutant", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    caught = False
    for pin in mlp_pins.ALL_MLP_PINS:
        try:
            pin(mod, oracle_lib)
        except AssertionError:
            caught = True
            break
    assert caught, f"no pin catches the mutant '{name}'"
