"""Planted mistakes in the CPU oracle: every one must fail at least one of the oracle's pins.

Each mutant is a copy of the oracle's C sources with one plausible mistake written in (a dropped
term, a wrong sign, scale or index, a transposed operand, gate and up swapped, an off-by-one in
the causal mask, a wrong rounding rule ...), compiled into a temporary library and loaded in place
of liboracle.so.  The pins of the function the mistake sits in (tests/test_oracle.py for the MLP,
LayerNorm and stack code, tests/test_oracle_attn.py for attention and the block,
tests/test_oracle_fp8.py for the E4M3 code) then run against it: a mutant that passed them all
would be a mistake the pins cannot see.  The unmodified copy passes every pin, which checks the
harness itself.  No GPU is involved; the mistakes are planted on the CPU only.
"""
import inspect
import itertools
import os
import shutil
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle
from oracle import build as oracle_build

import test_oracle
import test_oracle_attn
import test_oracle_fp8

CORE, ATTN, FP8 = "core", "attn", "fp8"
PIN_MODULES = {CORE: test_oracle, ATTN: test_oracle_attn, FP8: test_oracle_fp8}

# (name, group, source file, text, replacement, which occurrence: an index or None for every one)
MUTANTS = [
    # activations (oracle.c)
    ("gelu_scale", CORE, "oracle.c", "return 0.5 * z * (1.0 + erf(z / sqrt(2.0)));",
     "return 0.5 * z * (1.0 + erf(z / 2.0));", 0),
    ("gelu_grad_dropped_density_term", CORE, "oracle.c", "return cdf + z * pdf;", "return cdf;", 0),
    ("relu_grad_at_zero", CORE, "oracle.c", "case ORC_RELU: return z > 0.0 ? 1.0 : 0.0;",
     "case ORC_RELU: return z >= 0.0 ? 1.0 : 0.0;", 0),
    ("swiglu_missing_gate_factor", CORE, "oracle.c", "if (act == ORC_SWIGLU) return g * sigmoid(g) * u;",
     "if (act == ORC_SWIGLU) return sigmoid(g) * u;", 0),
    ("silu_grad_sign", CORE, "oracle.c", "u * s * (1.0 + g * (1.0 - s))", "u * s * (1.0 - g * (1.0 - s))", 0),
    ("swiglu_up_grad_missing_gate", CORE, "oracle.c", "if (act == ORC_SWIGLU) return g * sigmoid(g);",
     "if (act == ORC_SWIGLU) return sigmoid(g);", 0),
    # forward (oracle_core.inc)
    ("gate_up_swapped", CORE, "oracle_core.inc",
     "const int64_t gate_row = i * 2 * Fi + j, up_row = i * 2 * Fi + Fi + j;",
     "const int64_t gate_row = i * 2 * Fi + Fi + j, up_row = i * 2 * Fi + j;", 0),
    ("second_weight_transposed_in_shard", CORE, "oracle_core.inc",
     "WLD(B, ((f) / (Fi)) * (h) * (Fi) + (c) * (Fi) + ((f) % (Fi)))",
     "WLD(B, ((f) / (Fi)) * (h) * (Fi) + ((f) % (Fi)) * (h) + (c))", 0),
    ("shard_sum_keeps_last_partial", CORE, "oracle_core.inc", "        y[c] += p;", "        y[c] = p;", 0),
    ("row_subset_reads_wrong_row", CORE, "oracle_core.inc", "FN(fwd_row)(h, F, t, act, X + r * h,",
     "FN(fwd_row)(h, F, t, act, X + rr * h,", 0),
    # backward (oracle_core.inc)
    ("dx_drops_up_branch", CORE, "oracle_core.inc",
     "s += d1[f] * WLD(A, (i * 2 * Fi + j) * h + k) + d2[f] * WLD(A, (i * 2 * Fi + Fi + j) * h + k);",
     "s += d1[f] * WLD(A, (i * 2 * Fi + j) * h + k);", 0),
    ("da_without_activation_grad", CORE, "oracle_core.inc", "dg = coldh[r] * oracle_act_grad(act, colg[r]);",
     "dg = coldh[r];", 0),
    ("db_uses_preactivation", CORE, "oracle_core.inc",
     "const double hv = gated ? oracle_glu(act, colg[r], colu[r]) : oracle_act(act, colg[r]);",
     "const double hv = gated ? oracle_glu(act, colg[r], colu[r]) : colg[r];", 0),
    ("db_output_gradient_transposed", CORE, "oracle_core.inc",
     "for (int64_t c = 0; c < h; ++c) out[c] += ALD(gY, r * h + c) * hv;",
     "for (int64_t c = 0; c < h; ++c) out[c] += ALD(gY, r * h + (h - 1 - c)) * hv;", 0),
    # LayerNorm and the stack (oracle_core.inc, oracle.c)
    ("layernorm_unbiased_variance", CORE, "oracle_core.inc", "  var /= (double)h;",
     "  var /= (double)(h - 1);", 0),
    ("layernorm_eps_outside_root", CORE, "oracle_core.inc", "const double inv = 1.0 / sqrt(var + eps);",
     "const double inv = 1.0 / (sqrt(var) + eps);", 0),
    ("stack_layernorm_unbiased_variance", CORE, "oracle_core.inc", "  var /= (double)h;",
     "  var /= (double)(h - 1);", 1),
    ("stack_gated_up_row_is_gate_row", CORE, "oracle_core.inc",
     "if (gated) su += x[k] * WLD(A, (i * 2 * Fi + Fi + j) * h + k);",
     "if (gated) su += x[k] * WLD(A, (i * 2 * Fi + j) * h + k);", 0),
    ("stack_residual_dropped", CORE, "oracle.c", "for (int64_t k = 0; k < h; ++k) z[k] += y[k];",
     "for (int64_t k = 0; k < h; ++k) z[k] = y[k];", 0),
    ("stack_bwd_layernorm_term_sign", CORE, "oracle_core.inc", "g[k] += r * (gn[k] - mg - n[k] * mgn);",
     "g[k] += r * (gn[k] - mg + n[k] * mgn);", 0),
    ("stack_bwd_mean_term_dropped", CORE, "oracle_core.inc", "g[k] += r * (gn[k] - mg - n[k] * mgn);",
     "g[k] += r * (gn[k] - n[k] * mgn);", 0),
    ("stack_bwd_residual_gradient_dropped", CORE, "oracle_core.inc", "g[k] += r * (gn[k] - mg - n[k] * mgn);",
     "g[k] = r * (gn[k] - mg - n[k] * mgn);", 0),
    ("stack_bwd_db_transposed", CORE, "oracle_core.inc", "dB[(i * h + c) * Fi + j] += g[c] * hv;",
     "dB[(i * Fi + j) * h + c] += g[c] * hv;", 0),
    ("stack_bwd_da_up_uses_gate_grad", CORE, "oracle_core.inc",
     "dA[(i * 2 * Fi + Fi + j) * h + k] += d2[f] * x[k];", "dA[(i * 2 * Fi + Fi + j) * h + k] += d1[f] * x[k];",
     0),
    # attention and the block (oracle_attn.c)
    ("attn_scale_one_over_d", ATTN, "oracle_attn.c", "const double scale = 1.0 / sqrt((double)d);",
     "const double scale = 1.0 / (double)d;", 0),
    ("attn_mask_excludes_own_position", ATTN, "oracle_attn.c", "w[p] = s * scale;",
     "w[p] = (p == pos && pos > 0) ? -INFINITY : s * scale;", 0),
    ("attn_keys_from_value_rows", ATTN, "oracle_attn.c",
     "k[hd * d + e] = dot_w(h, x, Wi + (1 * nhi * d + j * d + e) * h);",
     "k[hd * d + e] = dot_w(h, x, Wi + (2 * nhi * d + j * d + e) * h);", 0),
    ("attn_output_weight_transposed", ATTN, "oracle_attn.c", "Wo[i * h * cols_i + c * cols_i + jj]",
     "Wo[i * h * cols_i + jj * h + c]", None),
    ("attn_softmax_not_normalised", ATTN, "oracle_attn.c", "o[hd * d + e] = acc / sum;", "o[hd * d + e] = acc;", 0),
    ("block_mlp_gate_up_swapped", ATTN, "oracle_attn.c", "const double g = dot_w(h, x, A + (i * 2 * Fi + j) * h);",
     "const double g = dot_w(h, x, A + (i * 2 * Fi + Fi + j) * h);", 0),
    # E4M3 (oracle_fp8.c)
    ("e4m3_ties_away_from_zero", FP8, "oracle_fp8.c", "double q = rint(ldexp(a, 3 - e));",
     "double q = round(ldexp(a, 3 - e));", 0),
    ("e4m3_exponent_bias_8", FP8, "oracle_fp8.c", "ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)", 0),
    ("e4m3_saturates_from_480", FP8, "oracle_fp8.c", "if (a >= 464.0) return sign | 0x7E;",
     "if (a >= 480.0) return sign | 0x7E;", 0),
    ("e4m3_subnormal_step", FP8, "oracle_fp8.c", "const double q = rint(a * 512.0);",
     "const double q = rint(a * 256.0);", 0),
    ("fp8_output_scale_missing", FP8, "oracle_fp8.c", "Y[rr * h + c] = sh * sb * s;", "Y[rr * h + c] = sb * s;", 0),
    ("fp8_requantise_without_scale", FP8, "oracle_fp8.c", "oracle_e4m3_encode((double)(float)(hv / sh))",
     "oracle_e4m3_encode((double)(float)hv)", 0),
]


def apply_mutation(text, old, new, which):
    count = text.count(old)
    assert count > 0, f"mutation site not found: {old}"
    if which is None:
        return text.replace(old, new)
    assert which < count, f"occurrence {which} of {count}: {old}"
    at = -1
    for _ in range(which + 1):
        at = text.index(old, at + 1)
    return text[:at] + new + text[at + len(old):]


def make_copy(root, name, mutation=None):
    d = os.path.join(root, name)
    os.makedirs(d)
    for f in oracle_build.SOURCES:
        shutil.copy(os.path.join(oracle_build.HERE, f), os.path.join(d, f))
    if mutation is not None:
        fname, old, new, which = mutation
        p = os.path.join(d, fname)
        with open(p, encoding="utf-8") as fh:
            text = fh.read()
        with open(p, "w", encoding="utf-8") as fh:
            fh.write(apply_mutation(text, old, new, which))
    return oracle_build.compile_library(d, os.path.join(d, "liboracle.so"))


def expand_pins(module):
    """(id, function, kwargs) for every pin of `module`, parametrisations expanded."""
    pins = []
    for name, fn in inspect.getmembers(module, inspect.isfunction):
        if not name.startswith("test_") or fn.__module__ != module.__name__:
            continue
        axes = []
        for mark in getattr(fn, "pytestmark", []):
            if mark.name != "parametrize":
                continue
            names = [a.strip() for a in mark.args[0].split(",")] if isinstance(mark.args[0], str) else list(mark.args[0])
            values = [v if len(names) > 1 else (v,) for v in mark.args[1]]
            axes.append([dict(zip(names, v)) for v in values])
        params = set(inspect.signature(fn).parameters)
        combos = [{}] if not axes else [dict(kv for d in c for kv in d.items()) for c in itertools.product(*axes)]
        for kw in combos:
            if set(kw) != params:
                break  # needs a fixture: not a plain pin
            pins.append((f"{name}{sorted(kw.items()) if kw else ''}", fn, kw))
    return pins


def failing_pins(lib_path, group, monkeypatch):
    """Ids of the pins of `group` that fail with the oracle library at `lib_path`."""
    monkeypatch.setattr(oracle, "_lib", None)
    monkeypatch.setattr(oracle._build, "build", lambda force=False: lib_path)
    failed = []
    for pid, fn, kw in expand_pins(PIN_MODULES[group]):
        try:
            fn(**kw)
        except Exception:  # an assertion, or the mutant rejecting a call
            failed.append(pid)
    monkeypatch.setattr(oracle, "_lib", None)
    return failed


@pytest.fixture(scope="module")
def libraries(tmp_path_factory):
    root = str(tmp_path_factory.mktemp("oracle_mutants"))
    jobs = {"unmodified": None}
    jobs.update({m[0]: m[2:] for m in MUTANTS})
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        futures = {name: ex.submit(make_copy, root, name, mut) for name, mut in jobs.items()}
        return {name: f.result() for name, f in futures.items()}


def test_mutant_names_unique():
    names = [m[0] for m in MUTANTS]
    assert len(names) == len(set(names))


@pytest.mark.parametrize("group", [CORE, ATTN, FP8])
def test_unmodified_copy_passes_every_pin(libraries, group, monkeypatch):
    assert failing_pins(libraries["unmodified"], group, monkeypatch) == []


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(libraries, mutant, monkeypatch):
    failed = failing_pins(libraries[mutant[0]], mutant[1], monkeypatch)
    assert failed, f"no pin sees the planted mistake {mutant[0]}"
