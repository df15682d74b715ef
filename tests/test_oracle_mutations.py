"""Plant plausible mistakes in a copy of the oracle (CPU only) and check that
the pins catch every one of them: a dropped term, a wrong sign, an
off-by-one boundary, a wrong index or a transposed operand."""

import os
import types

import pytest

import pins

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle", "bifocal.py")

# (name, text in oracle/bifocal.py, replacement)
MUTATIONS = [
    ("local boundary strict", "np.where(dist <= w0, s_abs, s_rem)",
     "np.where(dist < w0, s_abs, s_rem)"),
    ("G rounds down", "max(1, -(-L // w))", "max(1, L // w)"),
    ("G off by one", "max(1, -(-L // w))", "max(1, -(-L // w) + 1)"),
    ("rotation sign", "x1 * c - x2 * s, x2 * c + x1 * s", "x1 * c + x2 * s, x2 * c - x1 * s"),
    ("interleaved pairing", "x1, x2 = x[..., :h], x[..., h:]", "x1, x2 = x[..., 0::2], x[..., 1::2]"),
    ("alias is identity", "np.floor_divide(np.asarray(x, dtype=np.int64), int(G))",
     "np.asarray(x, dtype=np.int64)"),
    ("remote key not aliased", "k_rem = rnd(_rotate(xk, cos_t[fpos], sin_t[fpos]))",
     "k_rem = rnd(_rotate(xk, cos_t, sin_t))"),
    ("remote query not aliased", "q_rem = rnd(_rotate(xq, cos_t[fpos[rc]], sin_t[fpos[rc]]))",
     "q_rem = rnd(_rotate(xq, cos_t[rc], sin_t[rc]))"),
    ("frequency exponent", "-2.0 * i / d", "-1.0 * i / d"),
    ("no causal mask", "s = np.where(dist < 0, -np.inf, s)", "s = s"),
    ("lse drops the max", "(m + np.log(l))[..., 0]", "(np.log(l))[..., 0]"),
    ("scores unscaled", "s = scale * np.where(dist <= w0, s_abs, s_rem)",
     "s = np.where(dist <= w0, s_abs, s_rem)"),
    ("decode correction sign", "delta_k = alias(j, G) - j", "delta_k = j - alias(j, G)"),
    ("decode query position", "qp = L - 1\n", "qp = L\n"),
    ("decode local boundary", "local = (qp - j) <= w0", "local = (qp - j) < w0"),
    ("negative angle not transposed", "s = np.where((pos < 0)[..., None], -s, s)", "s = s"),
    ("angle composition bit test", "bit = ((mag >> j) & 1)", "bit = ((mag >> (j + 1)) & 1)"),
    ("three-pass sign", "- w_c[:, None] * o_c", "+ w_c[:, None] * o_c"),
    ("bf16 rounding keeps 7 bits", "quantum = np.ldexp(1.0, e - 8)", "quantum = np.ldexp(1.0, e - 7)"),
    ("chunk: cached keys not corrected", "rnd(rope_rotate(cached, alias(cpos, G) - cpos, theta))",
     "rnd(cached)"),
    ("chunk: query positions from zero", "qpos = np.arange(P0, Lt, dtype=np.int64)",
     "qpos = np.arange(0, C, dtype=np.int64)"),
    ("GQA heads interleaved", "            for h in range(hk * group, (hk + 1) * group):\n                rh",
     "            for h in range(hk, Hq, Hkv):\n                rh"),
    ("three-pass window strict", "window = causal & (dist <= w0)", "window = causal & (dist < w0)"),
    ("chunk: G from the chunk length", "    G = group_size(Lt, w_pretrained)", "    G = group_size(C, w_pretrained)"),
    ("decode: remote query at the absolute position", "q_rem = rope_rotate(xq, [alias(qp, G)], theta)[0]",
     "q_rem = rope_rotate(xq, [qp], theta)[0]"),
    ("decode: G from the cache capacity", "    G = group_size(L, w_pretrained)\n    if scale is None:\n        scale = 1.0 / math.sqrt(d)\n    qp",
     "    G = group_size(k_cache.shape[1], w_pretrained)\n    if scale is None:\n        scale = 1.0 / math.sqrt(d)\n    qp"),
]


def _mutant(old, new):
    src = open(ORACLE_SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    src = src.replace(old, new)
    mod = types.ModuleType("oracle_mutant")
    mod.__dict__["__name__"] = "oracle_mutant"
    exec(compile(src, "oracle_mutant.py", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(name, old, new):
    mod = _mutant(old, new)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(mod)
        except Exception as e:  # AssertionError, or the mutant crashing
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"mutation {name!r} passed every pin"
