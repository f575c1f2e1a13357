"""Plant plausible mistakes in a copy of the oracle and check that its pins fail.

Each entry replaces one fragment of an oracle file (a dropped term, a wrong
index, sign, operand or order) in a temporary copy of ``oracle/``, then runs
the pin file that covers it; the run must fail.  The mistakes live only in the
copy, on the CPU.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = {"scan.py": "tests/test_oracle_scan.py", "conv1d.py": "tests/test_oracle_conv_rms.py",
        "rmsnorm.py": "tests/test_oracle_conv_rms.py"}

MUTS = {
  "scan.py": [
    ("q uses h_t", "q = G * a_t * h_prev", "q = G * a_t * h_t"),
    ("dx drops ds*D", "dx[:, t] = ds * Dv[None, :] + d_t * GB", "dx[:, t] = d_t * GB"),
    ("dA drops delta", "dA += np.sum(q * d_t[:, :, None], axis=0)", "dA += np.sum(q, axis=0)"),
    ("G carried with a_t", "a_next = a_t\n", "a_next = avals[i - 1] if i > 0 else a_t\n"),
    ("dz uses silu not silu'", "dz[:, t] = dy_t * s_t * sig * (1.0 + z_t * (1.0 - sig))", "dz[:, t] = dy_t * s_t * sig * z_t"),
    ("dB drops x", "dB[:, t] = np.sum(G * (d_t * x_t)[:, :, None], axis=1)", "dB[:, t] = np.sum(G * d_t[:, :, None], axis=1)"),
    ("dC uses h_prev", "dC[:, t] = np.sum(ds[:, :, None] * h_t, axis=1)", "dC[:, t] = np.sum(ds[:, :, None] * h_prev, axis=1)"),
    ("exp sign", "a = np.exp(delta_t[:, :, None] * A[None, :, :])", "a = np.exp(-delta_t[:, :, None] * A[None, :, :])"),
    ("ddelta drops GB*x", "ddelta[:, t] = np.sum(q * A[None, :, :], axis=-1) + GB * x_t", "ddelta[:, t] = np.sum(q * A[None, :, :], axis=-1)"),
    ("gate on C.h only", "s = np.sum(h * Cm[:, t, None, :], axis=-1) + Dv[None, :] * x[:, t]\n        y[:, t] = s * (z[:, t] * _sigmoid(z[:, t]))",
     "s = np.sum(h * Cm[:, t, None, :], axis=-1)\n        y[:, t] = s * (z[:, t] * _sigmoid(z[:, t])) + Dv[None, :] * x[:, t]"),
    ("B and C swapped in y", "s = np.sum(h * Cm[:, t, None, :], axis=-1)", "s = np.sum(h * Bm[:, t, None, :], axis=-1)"),
    ("dh0 without a", "dh0 = a_next * G", "dh0 = G"),
    ("checkpoint after step", "            ckpt[:, t // chunk] = h\n        _, h = _step(h, delta[:, t], x[:, t], Bm[:, t], A)",
     "            pass\n        _, h = _step(h, delta[:, t], x[:, t], Bm[:, t], A)\n        if chunk and t % chunk == 0:\n            ckpt[:, t // chunk] = h"),
  ],
}
MUTS["conv1d.py"] = [
    ("tap order reversed", "        shift = K - 1 - k  # out[t] reads x[t - shift] through tap k", "        shift = k  # (mutated)"),
    ("fwd state shift", "    shift = K - 1 - k\n    out = np.zeros_like(x)", "    shift = k\n    out = np.zeros_like(x)"),
    ("db missing", "    db = np.sum(dout, axis=(0, 1))", "    db = np.zeros(D)"),
    ("dsilu without (1 - s)", "    return s * (1.0 + v * (1.0 - s))", "    return s * (1.0 + v * s)"),
    ("silu bwd uses act not pre", "    return conv1d_causal_bwd_ref(np.asarray(dact, np.float64) * dsilu_ref(pre), x, w)",
     "    return conv1d_causal_bwd_ref(np.asarray(dact, np.float64) * dsilu_ref(silu_ref(pre)), x, w)"),
    ("step tap order", "    new = np.concatenate([state[:, :, 1:], np.asarray(x_t, np.float64)[:, :, None]], axis=2)",
     "    new = np.concatenate([np.asarray(x_t, np.float64)[:, :, None], state[:, :, :-1]], axis=2)"),
]
MUTS["rmsnorm.py"] = [
    ("dot missing inv^2", "    dot = np.sum(dy * scale[None, :] * x, axis=1) * inv * inv", "    dot = np.sum(dy * scale[None, :] * x, axis=1) * inv"),
    ("dx drops /H", "    dx = inv[:, None] * (scale[None, :] * dy - x * dot[:, None] / H)", "    dx = inv[:, None] * (scale[None, :] * dy - x * dot[:, None])"),
    ("dscale drops inv", "    dscale = np.sum(dy * x * inv[:, None], axis=0)", "    dscale = np.sum(dy * x, axis=0)"),
    ("fwd eps outside root", "    rms = np.sqrt(np.mean(x * x, axis=1) + eps)", "    rms = np.sqrt(np.mean(x * x, axis=1)) + eps"),
    ("dx drops scale", "    dx = inv[:, None] * (scale[None, :] * dy - x * dot[:, None] / H)", "    dx = inv[:, None] * (dy - x * dot[:, None] / H)"),
]

CASES = [(f, n, a, b) for f, muts in MUTS.items() for (n, a, b) in muts]


@pytest.mark.parametrize("fname,name,frag,repl", CASES, ids=[f"{c[0]}:{c[1]}" for c in CASES])
def test_planted_mistake_fails_a_pin(tmp_path, fname, name, frag, repl):
    for d in ("oracle", "tests", "workloads"):
        shutil.copytree(os.path.join(ROOT, d), tmp_path / d, ignore=shutil.ignore_patterns("__pycache__", "golden"))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), tmp_path / "tests" / "golden")
    shutil.copy(os.path.join(ROOT, "pytest.ini"), tmp_path)
    p = tmp_path / "oracle" / fname
    s = p.read_text()
    assert s.count(frag) >= 1, f"fragment of '{name}' not found in oracle/{fname}"
    p.write_text(s.replace(frag, repl, 1))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", PINS[fname]],
                       cwd=tmp_path, capture_output=True, text=True, env=dict(os.environ, PYTHONPATH=str(tmp_path)))
    assert r.returncode != 0, f"no pin caught '{name}' in oracle/{fname}"
