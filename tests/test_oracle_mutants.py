"""Plausible mistakes planted in a copy of the oracle (on the CPU) must each fail a pin.

Each mutant is the oracle's C source with one textual change, compiled into a temporary
library and swapped in for the real one while the pins run."""
import ctypes
import os
import subprocess

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "decay_scales_columns": ("Si[j] *= al[i];", "Si[j] *= al[j];"),
    "beta_dropped": ("u[j] = beta * (v[j] - u[j]);", "u[j] = (v[j] - u[j]);"),
    "delta_sign_flipped": ("u[j] = beta * (v[j] - u[j]);", "u[j] = beta * (v[j] + u[j]);"),
    "readout_transposed": ("u[j] += Si[j] * k[i];", "u[j] += S[(int64_t)j * d + i] * k[i];"),
    "outer_product_transposed": ("Si[j] += k[i] * u[j];", "Si[j] += k[j] * u[i];"),
    "output_reads_key": ("o[j] += Si[j] * q[i];", "o[j] += Si[j] * k[i];"),
    "decay_base_two": ("al[i] = exp((double)a->g[base + i]);", "al[i] = exp2((double)a->g[base + i]);"),
    "checkpoint_off_by_one": ("a->ckpt_pos[c] == t + 1", "a->ckpt_pos[c] == t + 2"),
    "initial_state_ignored": ("S[e] = (double)s0[e];", "S[e] = 0.0 * (double)s0[e];"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    inc = os.path.dirname(oracle.__file__)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", f"-I{inc}",
                    "-o", str(so), str(path), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    lib.kda_ref_run.restype = ctypes.c_int
    lib.kda_ref_run.argtypes = [ctypes.POINTER(oracle._Args), ctypes.POINTER(ctypes.c_int)]
    return lib


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name, monkeypatch):
    old, new = MUTANTS[name]
    lib = _build_mutant(tmp_path, name, old, new)
    oracle._load()
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin()
        except (AssertionError, oracle.OracleError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"


# The output epilogue ("Kimi K3.1 Pro 架构完全拆解" section 3.3) is plain numpy: each mutant
# is the module's source with one textual change, loaded in place of the real module.
EPILOGUE_MUTANTS = {
    "rms_uses_sum": ("np.mean(o * o, axis=-1, keepdims=True)", "np.sum(o * o, axis=-1, keepdims=True)"),
    "rms_without_sqrt": ("np.sqrt(ms + eps)", "(ms + eps)"),
    "eps_outside_sqrt": ("np.sqrt(ms + eps)", "(np.sqrt(ms) + eps)"),
    "gate_not_sigmoid": ("return sigmoid(a) * g * o", "return a * g * o"),
    "gamma_dropped": ("return sigmoid(a) * g * o", "return sigmoid(a) * o"),
}


@pytest.mark.parametrize("name", sorted(EPILOGUE_MUTANTS))
def test_epilogue_mutant_is_caught(name, monkeypatch):
    import sys
    import types
    import oracle.epilogue as real
    old, new = EPILOGUE_MUTANTS[name]
    src = open(real.__file__).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mod = types.ModuleType("oracle.epilogue")
    exec(compile(src.replace(old, new), real.__file__, "exec"), mod.__dict__)
    monkeypatch.setitem(sys.modules, "oracle.epilogue", mod)
    caught = []
    for pin in (oracle_pins.pin_epilogue_hand_values, oracle_pins.pin_epilogue_invariants,
                oracle_pins.pin_epilogue_eps_closed_form):
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"


FRONTEND_MUTANTS = {
    "taps_reversed": ("y[..., i, :] += w[:, j] * full[..., W - 1 + i - j, :]",
                      "y[..., i, :] += w[:, W - 1 - j] * full[..., W - 1 + i - j, :]"),
    "conv_reads_ahead": ("full[..., W - 1 + i - j, :]", "full[..., min(W - 1 + i + j, full.shape[-2] - 1), :]"),
    "silu_is_sigmoid": ("return x * sigmoid(x)", "return sigmoid(x)"),
    "l2_without_sqrt": ("n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))", "n = np.sum(x * x, axis=-1, keepdims=True)"),
    "gate_without_exp_scale": ("sigmoid(np.exp(np.asarray(a_log, np.float64)) * np.asarray(z, np.float64))",
                               "sigmoid(np.asarray(a_log, np.float64) * np.asarray(z, np.float64))"),
    "beta_raw": ("def beta_gate(b):\n    return sigmoid(b)", "def beta_gate(b):\n    return np.asarray(b, np.float64)"),
    "cache_keeps_oldest": ("return full[..., full.shape[-2] - keep:, :]", "return full[..., :keep, :]"),
    "decay_dropped": ("S = np.exp(g[:, i])[..., :, None] * S", "S = S"),
    "k_not_normalised": ("k = l2_normalize(streams[1])", "k = streams[1]"),
}


@pytest.mark.parametrize("name", sorted(FRONTEND_MUTANTS))
def test_frontend_mutant_is_caught(name, monkeypatch):
    import sys
    import types
    import oracle.frontend as real
    old, new = FRONTEND_MUTANTS[name]
    src = open(real.__file__).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mod = types.ModuleType("oracle.frontend")
    mod.__package__ = "oracle"
    exec(compile(src.replace(old, new), real.__file__, "exec"), mod.__dict__)
    monkeypatch.setitem(sys.modules, "oracle.frontend", mod)
    caught = []
    for pin in (oracle_pins.pin_frontend_conv_against_numpy, oracle_pins.pin_frontend_silu_and_l2,
                oracle_pins.pin_frontend_gates, oracle_pins.pin_frontend_replay_identities,
                oracle_pins.pin_frontend_recurrence_against_c_oracle, oracle_pins.pin_frontend_step_retrieval):
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
