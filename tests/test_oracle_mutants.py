"""The oracle's pins catch plausible mistakes (CPU only).

Each mutant below is the oracle's C++ source with one plausible mistake
planted in it: a dropped term, a wrong sign, a wrong or transposed index, a
wrong normalisation, the wrong operand, another padding.  Every mutant is
compiled into a separate copy of the oracle package and the pins of
``test_oracle_pins.py`` are run against it; at least one pin must fail.  The
unmodified source, built the same way, must pass every pin (the control).

Every mutant keeps all array accesses in bounds, so a mutant can give wrong
numbers but cannot crash the test process.
"""
import importlib.util
import os
import shutil
from concurrent.futures import ThreadPoolExecutor

import test_oracle_pins as pins

ORACLE_DIR = os.path.dirname(os.path.abspath(pins.oracle.__file__))

# (name, original text, planted text, which occurrence of the original: None = the only one)
MUTANTS = [
    # Haar pair
    ("analysis normalisation 1/4", "out[((size_t)b * Hh + p) * Wh + q] = 0.5 * s;",
     "out[((size_t)b * Hh + p) * Wh + q] = 0.25 * s;", None),
    ("column-high band signed by the row bit", "else if (b == 2) parity = v;", "else if (b == 2) parity = u;", None),
    ("synthesis signs transposed", "s += band_sign(b, u, v) * in[", "s += band_sign(b, v, u) * in[", None),
    ("replicate instead of zero padding", "(i < H && j < W) ? in[(size_t)i * W + j] : 0.0",
     "in[(size_t)(i < H ? i : H - 1) * W + (j < W ? j : W - 1)]", None),
    # forward cascade
    ("kernel taps transposed", "s += w[du * K + dv] * in[(size_t)ii * W + jj];",
     "s += w[dv * K + du] * in[(size_t)ii * W + jj];", None),
    ("convolution instead of cross-correlation", "const int ii = i + du - r, jj = j + dv - r;",
     "const int ii = i - du + r, jj = j - dv + r;", 0),  # conv_same: the first of three
    ("convolved low-pass feeds the next level", "cur.assign(Y.begin(), Y.begin() + g.plane(l));",
     "cur.assign(Z[l].begin(), Z[l].begin() + g.plane(l));", None),
    ("coarser reconstruction not added", "for (size_t t = 0; t < g.plane(l); ++t) Zl[t] += next[t];",
     "for (size_t t = 0; t < g.plane(l); ++t) Zl[t] += 0.0;", None),
    ("wavelet scale pass dropped", "for (size_t t = 0; t < g.plane(l); ++t) zb[t] *= s;",
     "for (size_t t = 0; t < g.plane(l); ++t) zb[t] *= 1.0;", None),
    ("bias outside the base scale", "y[t] = sb * (base[t] + bias) + next[t];",
     "y[t] = sb * base[t] + bias + next[t];", None),
    # backward cascade
    ("base-scale gradient without the bias term", "*dsb += dot(P.wb(c), Gb.data(), KK) + P.bias(c) * gsum;",
     "*dsb += dot(P.wb(c), Gb.data(), KK);", None),
    ("bias gradient without the base scale", "if (db) *db += sb * gsum;", "if (db) *db += gsum;", None),
    ("sub-band weight gradient without the scale", "dw_sub_c[((size_t)(l - 1) * 4 + b) * KK + t] += s * G[t];",
     "dw_sub_c[((size_t)(l - 1) * 4 + b) * KK + t] += G[t];", None),
    ("wavelet-scale gradient against the unconvolved band",
     "dsw_c[(l - 1) * 4 + b] += dot(gzb, Cv[l].data() + b * g.plane(l), g.plane(l));",
     "dsw_c[(l - 1) * 4 + b] += dot(gzb, Y[l].data() + b * g.plane(l), g.plane(l));", None),
    ("band adjoint without the scale", "P.ws(l, c, b), K, s, gY[l].data()", "P.ws(l, c, b), K, 1.0, gY[l].data()", None),
    ("adjoint taps transposed", "out[(size_t)ii * W + jj] += w[du * K + dv] * gv;",
     "out[(size_t)ii * W + jj] += w[dv * K + du] * gv;", None),
    ("weight gradient with flipped offsets", "const int ii = i + du - r, jj = j + dv - r;",
     "const int ii = i - du + r, jj = j - dv + r;", 2),  # conv_same_weight_grad_add
    ("analysis-chain adjoint drops the coarser levels", "for (size_t t = 0; t < g.plane(l); ++t) gYt[t] += acc[t];",
     "for (size_t t = 0; t < g.plane(l); ++t) gYt[t] += 0.0;", None),
    # direct form
    ("direct coefficients normalised by 4^-l", "const double norm = std::ldexp(1.0, -l);",
     "const double norm = std::ldexp(1.0, -2 * l);", None),
    ("closed-form synthesis reads bit l", "const int u = bit(i, l - 1), v = bit(j, l - 1);",
     "const int u = bit(i, l), v = bit(j, l);", None),
    ("closed-form synthesis without 2^-l", "acc += std::ldexp(1.0, -l) * s;", "acc += s;", None),
    ("direct wavelet-scale gradient against the scale", "dsw_c[(l - 1) * 4 + b] += P.ws(l, c, b)[du * K + dv] * G;",
     "dsw_c[(l - 1) * 4 + b] += P.sw(l, c, b) * G;", None),
]

S = pins.SHAPES
PINS = [  # (name, call): quick members of each pin family
    ("perfect reconstruction", lambda: [pins.test_perfect_reconstruction(h, w) for h, w in [(7, 7), (8, 5), (1, 5)]]),
    ("parseval", lambda: pins.test_parseval(7, 9)),
    ("synthesis = analysis^T", lambda: pins.test_synthesis_is_transpose_of_analysis()),
    ("haar golden", lambda: pins.test_haar_golden_2x2()),
    ("delta golden", lambda: [pins.test_delta_kernel_golden(c, f) for c in ("caseA", "caseB", "caseC")
                              for f in ("cascade", "direct")]),
    ("delta closed form", lambda: [pins.test_delta_kernel_closed_form(7, 9, 3, k) for k in (3, 5)]),
    ("single-band projections", lambda: [pins.test_single_band_projection_level1(b) for b in range(4)]),
    ("coarsest low-pass block mean", lambda: pins.test_coarsest_lowpass_is_block_mean()),
    ("base path = grouped conv", lambda: pins.test_base_path_equals_grouped_conv()),
    ("forward = torch composition", lambda: [pins.test_forward_equals_torch_composition(s) for s in S]),
    ("backward = torch autograd", lambda: [pins.test_backward_equals_torch_autograd(s, b) for s in S[:4]
                                           for b in (True, False)]),
    ("cascade = direct", lambda: [pins.test_cascade_equals_direct(h, w, L) for h, w, L in
                                  [(5, 9, 3), (4, 4, 2), (7, 7, 1), (8, 6, 4)]]),
    ("linearity", lambda: pins.test_linearity_in_x()),
    ("adjoint identity", lambda: [pins.test_adjoint_identity(s) for s in [(2, 2, 11, 9, 3, 5), (1, 1, 7, 5, 5, 7)]]),
    ("finite differences, parameters", lambda: pins.test_finite_difference_every_parameter()),
    ("finite differences, dx", lambda: pins.test_finite_difference_dx_sample()),
]


def plant(src, old, new, occurrence):
    parts = src.split(old)
    if occurrence is None:
        assert len(parts) == 2, f"{old!r} occurs {len(parts) - 1} times"
        occurrence = 0
    assert len(parts) > occurrence + 1, f"{old!r} has no occurrence {occurrence}"
    return old.join(parts[:occurrence + 1]) + new + old.join(parts[occurrence + 1:])


def make_variant(root, name, src):
    """A copy of the oracle package with `src` as its C++ source, compiled."""
    pkg = os.path.join(root, name)
    os.makedirs(pkg)
    shutil.copy(os.path.join(ORACLE_DIR, "__init__.py"), os.path.join(pkg, "__init__.py"))
    with open(os.path.join(pkg, "wtconv_oracle.cpp"), "w") as f:
        f.write(src)
    spec = importlib.util.spec_from_file_location(name, os.path.join(pkg, "__init__.py"),
                                                  submodule_search_locations=[pkg])
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    return mod


def first_failing_pin(monkeypatch, mod):
    monkeypatch.setattr(pins, "oracle", mod)  # undone at teardown
    for name, call in PINS:
        try:
            call()
        except (AssertionError, ValueError):
            return name
    return None


def test_every_planted_mistake_fails_a_pin(tmp_path, monkeypatch):
    with open(os.path.join(ORACLE_DIR, "wtconv_oracle.cpp")) as f:
        src = f.read()
    sources = [("control", src)] + [(f"mutant{i}", plant(src, old, new, occ))
                                    for i, (_, old, new, occ) in enumerate(MUTANTS)]
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:  # g++ runs in parallel
        mods = list(ex.map(lambda a: make_variant(str(tmp_path), *a), sources))
    control, mutants = mods[0], mods[1:]
    # the control passes every pin, so a failure below is the planted mistake's
    assert first_failing_pin(monkeypatch, control) is None
    caught = {what: first_failing_pin(monkeypatch, mod) for (what, *_), mod in zip(MUTANTS, mutants)}
    for what, pin in caught.items():
        print(f"{what:55s} -> {pin}")
    missed = [what for what, pin in caught.items() if pin is None]
    assert not missed, f"no pin fails for: {missed}"
