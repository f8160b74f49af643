"""The oracle's pins catch plausible mistakes.

Each case copies ``oracle/``, ``gen/`` and ``tests/`` into a temporary
directory, plants one typical slip in the copy of the oracle (a dropped or
flipped term, a wrong rounding direction, an index off by one, a transposed
grouping, a wrong tie order) and runs the pin tests of that oracle module on
the copy: they must fail.  An unmodified copy must pass, so a failure is due
to the planted mistake and not to the copying.  CPU only; the mistakes live
only in the temporary copy.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PINS = {
    "quant": ["tests/test_oracle_quant.py"],
    "select": ["tests/test_oracle_select.py", "tests/test_oracle_select_heads.py"],
    "attention": ["tests/test_oracle_attention.py"],
    "prefill": ["tests/test_oracle_prefill.py"],
    "accounting": ["tests/test_oracle_accounting.py"],
}

# (oracle module, original text, planted mistake, name)
MUTATIONS = [
    ("quant", "xg = x.reshape(x.shape[:-1] + (d // group, group))",
     "xg = np.swapaxes(x.reshape(x.shape[:-1] + (group, d // group)), -1, -2)", "strided groups"),
    ("quant", "zero = mn.astype(np.float16)", "zero = mx.astype(np.float16)", "zero point = max"),
    ("quant", "scale = min_step_fp16(mx, mn, qmax)",
     "scale = ((mx - mn) / float(qmax)).astype(np.float16)", "scale rounded to nearest"),
    ("quant", "c = np.where(dn & ((d < 0) | ((d == 0) & (c % 2 == 1))), c - 1, c)",
     "c = np.where(dn & (d <= 0), c - 1, c)", "ties always to the lower code"),
    ("quant", "d = x - (z + (c - 0.5) * s)            # against the midpoint below c",
     "d = x - (z + c * s)", "truncated codes"),
    ("quant", "return (cg * s + z).reshape(codes.shape)", "return (cg * s - z).reshape(codes.shape)",
     "dequantise sign"),
    ("select", "k = -((-P * int(rho_ppm)) // 1_000_000)", "k = (P * int(rho_ppm)) // 1_000_000",
     "k rounded down"),
    ("select", "return q.reshape(B, num_kv_heads, g, T, d).sum(axis=(2, 3))",
     "return q.reshape(B, g, num_kv_heads, T, d).sum(axis=(1, 3))", "GQA grouping transposed"),
    ("select", "order = np.lexsort((pos, -flat[r]))", "order = np.lexsort((-pos, -flat[r]))",
     "ties to the higher index"),
    ("select", "return max(0, int(L) - int(window))", "return max(0, int(L) - int(window) - 1)",
     "prefix length off by one"),
    ("select", "z = a * (Q @ k[b, kh, :L].T)", "z = a * (Q @ k[b, kh, :P].T)",
     "mass softmax over the prefix only"),
    ("select", "z = a * (Q @ k[b, kh, :L].T)", "z = (Q @ k[b, kh, :L].T)", "mass logits without alpha"),
    ("select", "A = e / e.sum(axis=1, keepdims=True)                  # softmax over the L keys",
     "A = e / e.sum(axis=0, keepdims=True)                  # softmax over the L keys",
     "mass normalised over the rows"),
    ("select", "u = q.sum(axis=2).reshape(B, HKV, g, d)", "u = q.sum(axis=2).reshape(B, g, HKV, d).swapaxes(1, 2)",
     "query head to KV head strided"),
    ("select", "order = np.lexsort((rest, -np.asarray(S_group, dtype=np.float64)[rest]))",
     "order = np.lexsort((rest, np.asarray(S_group, dtype=np.float64)[rest]))", "fill by the lowest group score"),
    ("select", "u = q.sum(axis=2).reshape(B, HKV, g, d)", "u = q[:, :, -1].reshape(B, HKV, g, d)",
     "head score from one proxy"),
    ("select", "Q = q[b, kh * g:(kh + 1) * g].reshape(g * T, d)", "Q = q[b, kh::HKV].reshape(g * T, d)",
     "mass GQA grouping strided"),
    ("attention", "a = 1.0 / math.sqrt(d) if alpha is None else alpha",
     "a = 1.0 / d if alpha is None else alpha", "alpha = 1/d"),
    ("attention", "K[:, :, :P, :] = np.where(keep[..., None], K[:, :, :P, :], Kq)",
     "K[:, :, :P, :] = Kq", "vertical lines quantised too"),
    ("attention", "l = sum(s[1] * np.exp(s[0] - m) for s in states)",
     "l = sum(s[1] * np.exp(m - s[0]) for s in states)", "merge rescale sign"),
    ("attention", "for seg in (vl, np.arange(max(P, 0), L)):",
     "for seg in (vl, np.arange(max(P, 0) + 1, L)):", "tail segment off by one"),
    ("attention", "logits = alpha * (q @ K.T)", "logits = alpha * (q @ K.T) * 1.0001",
     "perturbed logit scale"),
    ("attention", "Vq = fake_quant(V[:, :, :P, :], bits if bits_v is None else bits_v)",
     "Vq = fake_quant(V[:, :, :P, :], bits)", "values quantised at the key width"),
    ("prefill", '"fp4": 6.0}', '"fp4": 4.0}', "FP4 c_B"),
    ("prefill", "vals = [m * 0.5 if e == 0 else", "vals = [m * 0.25 if e == 0 else", "e2m1 subnormal step"),
    ("prefill", "lg = np.where(pos[None, :] <= rows[:, None], lg, -np.inf)",
     "lg = np.where(pos[None, :] < rows[:, None] + 2, lg, -np.inf)", "causal mask off by one"),
    ("prefill", "alpha * qb @ Kall[nq:].T], axis=1)", "alpha * qhat @ Kall[nq:].T], axis=1)",
     "BF16 branch uses quantised queries"),
    ("prefill", "d = a - mids[np.maximum(i - 1, 0)] * s",
     "d = a - grid[np.maximum(i, 0)] * s", "codes truncated toward zero"),
    ("prefill", "i = np.where((i > 0) & ((d < 0) | ((d == 0) & (i % 2 == 1))), i - 1, i)",
     "i = np.where((i > 0) & (d <= 0), i - 1, i)", "ties toward zero"),
    ("prefill", "vq[t0:t0 + len(j)] = quantize_symmetric(v[b, kh, j], None, dtype)[0]",
     "vq[t0:t0 + len(j)] = quantize_symmetric(v[b, kh, j], 0, dtype)[0]", "V scales per channel"),
    ("prefill", "s = (amax / np.float32(C_B[dtype])).astype(np.float32)",
     "s = (amax / np.float32(C_B[dtype] + 1)).astype(np.float32)", "c_B off by one"),
    ("prefill", "inb = (bpos[None, :] > lim[:, None])", "inb = (bpos[None, :] >= lim[:, None])",
     "band includes i - W"),
    ("prefill", "lg = np.where(pos[None, :] <= lim[:, None], lg, -np.inf)",
     "lg = np.where(pos[None, :] <= rows[:, None], lg, -np.inf)", "band: quantised keys up to i"),
    ("prefill", "& (bpos[None, :] <= rows[:, None])", "& (bpos[None, :] < rows[:, None])",
     "band leaves out the query's own key"),
    ("accounting", "return d // 2 + ((d // group) * 4 if with_meta else 0)",
     "return d // 2 + ((d // group) * 2 if with_meta else 0)", "metadata bytes halved"),
]


def _copy_tree(dst):
    for sub in ("oracle", "gen", "tests"):
        shutil.copytree(os.path.join(ROOT, sub), os.path.join(dst, sub),
                        ignore=shutil.ignore_patterns("__pycache__"))


def _run_pins(workdir, module):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu", *PINS[module]],
                       cwd=workdir, capture_output=True, text=True, env=env, timeout=600)
    return r.returncode, r.stdout[-2000:]


def _mutant(base, i):
    module, old, new, name = MUTATIONS[i]
    wd = os.path.join(base, f"m{i}")
    _copy_tree(wd)
    path = os.path.join(wd, "oracle", module + ".py")
    src = open(path).read()
    assert src.count(old) == 1, f"mutation target for '{name}' not found once in oracle/{module}.py"
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    rc, out = _run_pins(wd, module)
    return name, rc, out


def test_unmodified_copy_passes(tmp_path):
    _copy_tree(str(tmp_path))
    for module in PINS:
        rc, out = _run_pins(str(tmp_path), module)
        assert rc == 0, f"pins of oracle/{module}.py fail on an unmodified copy:\n{out}"


def test_every_planted_mistake_is_caught(tmp_path):
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(lambda i: _mutant(str(tmp_path), i), range(len(MUTATIONS))))
    missed = [name for name, rc, _ in results if rc == 0]
    broken = [(name, out) for name, rc, out in results if rc not in (0, 1)]
    assert not broken, f"pytest did not run cleanly for: {broken}"
    assert not missed, f"planted mistakes not caught by the pins: {missed}"


@pytest.mark.parametrize("module", sorted(PINS))
def test_each_module_has_mutations(module):
    assert any(m[0] == module for m in MUTATIONS)
