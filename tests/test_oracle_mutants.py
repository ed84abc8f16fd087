"""The pins have teeth: each plausible mistake planted in a copy of the
oracle's C source must make at least one pin of test_oracle_pins fail.

Mistakes are planted in the oracle only, on the CPU; the oracle's own source
file is never modified.
"""

import inspect

import pytest

import oracle
from tests import test_oracle_pins as pins

# (name, text in moe_oracle.c, replacement)
MUTANTS = [
    ("weights gathered from biased scores", "double wj = s[order[j]];", "double wj = cb[order[j]];"),
    ("ties go to the higher index", "(cb[order[j - 1]] < cb[e])", "(cb[order[j - 1]] <= cb[e])"),
    ("ascending selection", "(cb[order[j - 1]] < cb[e])", "(cb[order[j - 1]] > cb[e])"),
    ("bias added to the logit", "cb[e] = s[e] + (bias ? (double)bias[e] : 0.0);",
     "cb[e] = sigmoid(l[e] + (bias ? (double)bias[e] : 0.0));"),
    ("bias dropped from selection", "cb[e] = s[e] + (bias ? (double)bias[e] : 0.0);", "cb[e] = s[e];"),
    ("scale applied before the norm", "if (c->route_norm) wj = wj / sum;\n            wj = wj * c->route_scale;",
     "wj = wj * c->route_scale;\n            if (c->route_norm) wj = wj / (sum * c->route_scale) * c->route_scale * c->route_scale;"),
    ("norm ignores route_norm", "if (c->route_norm) wj = wj / sum;", "wj = wj / sum;"),
    ("sigmoid sign flipped", "return 1.0 / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(z));"),
    ("softmax without normaliser", "s[e] = exp(l[e] - m) / z;", "s[e] = exp(l[e] - m);"),
    ("gate clamped from below too", "double gc = g > c->limit ? c->limit : g;",
     "double gc = g > c->limit ? c->limit : (g < -c->limit ? -c->limit : g);"),
    ("up not clamped", "double uc = u > c->limit ? c->limit : (u < -c->limit ? -c->limit : u);",
     "double uc = u;"),
    ("beta dropped", "(uc + c->beta)", "(uc)"),
    ("alpha dropped", "sigmoid(c->alpha * gc)", "sigmoid(gc)"),
    ("silu on the up projection", "return g * sigmoid(g) * u;", "return g * sigmoid(u) * u;"),
    ("down projection transposed", "wget(Wd, sd, wd, (size_t)h, (size_t)i, (size_t)H, (size_t)W)",
     "wget(Wd, sd, wd, (size_t)i, (size_t)h, (size_t)W, (size_t)H)"),
    ("gate/up swapped", "gi += wget(Wg, sg, wd,", "gi += wget(Wu, su, wd,"),
    ("router weight transposed", "(double)Wr[(size_t)e * H + h]", "(double)Wr[(size_t)h * E + e]"),
    ("shared expert scaled by route_scale", "for (int h = 0; h < H; h++) y[h] += 1.0 * ye[h];",
     "for (int h = 0; h < H; h++) y[h] += c->route_scale * ye[h];"),
    ("packed shared read from slice 0", "(size_t)idx[s] : (size_t)c->E;", "(size_t)idx[s] : (size_t)0;"),
    ("packed shared scaled by route_scale", "w[s] : 1.0;", "w[s] : c->route_scale;"),
    ("shared expert dropped", "if (!c->shared_packed && c->S > 0) {\n        expert_mlp", "if (0) {\n        expert_mlp"),
    ("one routed slot dropped", "for (int s = 0; s <= k; s++) {", "for (int s = 1; s <= k; s++) {"),
    ("margin off by one", "cb[order[k - 1]] - cb[order[k]]", "cb[order[k - 2 < 0 ? 0 : k - 2]] - cb[order[k]]"),
    ("bf16 decoded with the wrong shift", "<< 16;", "<< 15;"),
    # the layers around the block
    ("dense MLP reads the routed width", "j->sc[4], j->sc[5], c->S, NULL, NULL, NULL,\n               j->Y",
     "j->sc[4], j->sc[5], c->S / 2, NULL, NULL, NULL,\n               j->Y"),
    ("rmsnorm without eps", "sqrt(ss / (double)H + eps)", "sqrt(ss / (double)H)"),
    ("rmsnorm over H - 1", "sqrt(ss / (double)H + eps)", "sqrt(ss / (double)(H - 1) + eps)"),
    ("rmsnorm by the mean square, not its root", "const double r = sqrt(ss / (double)H + eps);",
     "const double r = ss / (double)H + eps;"),
    ("Gemma norm without the + 1", "(gemma ? 1.0 + w[h] : w[h])", "(gemma ? w[h] : w[h])"),
    ("norm weight ignored", "(gemma ? 1.0 + w[h] : w[h])", "(gemma ? 1.0 + w[h] : 1.0)"),
    # block-scaled expert weights
    ("MX scales read row-major", "scale[(c / 32) * rows + r]", "scale[r * (cols / 32) + c / 32]"),
    ("E4M3 exponent bias 8", "ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    ("E4M3 subnormals decoded as normals", "e == 0 ? ldexp((double)m / 8.0, -6)", "e == 0 ? ldexp(1.0 + (double)m / 8.0, -7)"),
    ("E4M3 mantissa of 2 bits", "(double)m / 8.0, e - 7", "(double)m / 4.0, e - 7"),
    ("E2M1 nibbles swapped", "(i & 1) ? b >> 4 : b & 15", "(i & 1) ? b & 15 : b >> 4"),
    ("E2M1 exponent bias 0", "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e)"),
    ("E8M0 bias 128", "ldexp(1.0, (int)s - 127)", "ldexp(1.0, (int)s - 128)"),
    ("MX block of 16", "scale[(c / 32) * rows + r]", "scale[(c / 16) * rows + r]"),
    ("MX scale of the up projection used for gate", "gi += wget(Wg, sg, wd,", "gi += wget(Wg, su, wd,"),
]

PIN_TESTS = [(name, fn) for name, fn in inspect.getmembers(pins, inspect.isfunction)
             if name.startswith("test_") and name != "test_margin_filter_drives_generator_redraws"]


def _param_sets(fn):
    """Expand the pytest.mark.parametrize marks of a pin into argument dicts."""
    marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
    sets = [{}]
    for m in marks:
        names = [n.strip() for n in m.args[0].split(",")]
        new = []
        for s in sets:
            for vals in m.args[1]:
                vals = vals if isinstance(vals, (tuple, list)) else (vals,)
                new.append({**s, **dict(zip(names, vals))})
        sets = new
    return sets


def _some_pin_fails() -> bool:
    for _, fn in PIN_TESTS:
        for kw in _param_sets(fn):
            try:
                fn(**kw)
            except Exception:
                return True
    return False


def test_unmutated_source_passes_every_pin(tmp_path):
    path = oracle.compile_variant(oracle.source_text(), str(tmp_path / "lib_ok.so"))
    with oracle.using_library(path):
        assert not _some_pin_fails()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = oracle.source_text()
    assert src.count(old) >= 1, f"mutant anchor not found: {old!r}"
    path = oracle.compile_variant(src.replace(old, new), str(tmp_path / "lib_mut.so"))
    with oracle.using_library(path):
        assert _some_pin_fails(), f"no pin caught: {name}"
