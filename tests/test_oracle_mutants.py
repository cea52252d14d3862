"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one of them.  Each mutant is compiled to a temporary library and
its pins run in a subprocess, so an out-of-range access in a mutant shows up
as a failure rather than taking down the test run."""
import os
import subprocess
import sys
import tempfile

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, text in dopt_oracle.c, replacement)
MUTANTS = [
    ("no_scale_first_rank", "float part = scale * orc_grad(grads, grad_type, first, idx);",
     "float part = orc_grad(grads, grad_type, first, idx);"),
    ("skip_last_rank", "for (int32_t q = first + 1; q < first + R; ++q) {",
     "for (int32_t q = first + 1; q < first + R - 1; ++q) {"),
    ("skip_last_instance", "for (int32_t inst = 0; inst < instances; ++inst) {\n        int32_t first",
     "for (int32_t inst = 0; inst < instances - 1 || inst == 0; ++inst) {\n        int32_t first"),
    ("writeback_first_instance_only",
     "for (int32_t inst = 0; inst < instances; ++inst)\n                        params[inst * R + r][bi - w0] = updated;",
     "params[r][bi - w0] = updated;"),
    ("update_sign", "ww = ww - delta;", "ww = ww + delta;"),
    ("no_bias_correction1", "s.step_size = (float)(lr / (1.0 - pow(b1, (double)t)));",
     "s.step_size = (float)lr;"),
    ("no_bias_correction2", "s.bc2_sqrt = (float)sqrt(1.0 - pow(b2, (double)t));",
     "s.bc2_sqrt = 1.0f;"),
    ("eps_inside_sqrt", "float root = sqrtf(vv);", "float root = sqrtf(vv + s->eps);"),
    ("m_uses_beta2", "float t1 = s->b1 * mm;", "float t1 = s->b2 * mm;"),
    ("m_uses_one_minus_beta2", "float t2 = s->one_minus_b1 * g;", "float t2 = s->one_minus_b2 * g;"),
    ("v_not_squared", "float gg = g * g;", "float gg = g;"),
    ("no_weight_decay", "ww = ww * s->decay;", "ww = ww;"),
    ("decay_sign", "s.decay = (float)(1.0 - lr * wd);", "s.decay = (float)(1.0 + lr * wd);"),
    ("wd_ignores_mask", "int decays = wd_mask ? (wd_mask[p] != 0) : 1;", "int decays = 1;"),
    ("grad_via_bucket_range", "float g = shard[pc->gbuf_local.start + t];",
     "float g = shard[pc->gbuf_world_in_bucket.start + t];"),
    ("master_via_local_range", "int64_t mi = pstart[p] + pc->param.start + t;",
     "int64_t mi = pstart[p] + pc->gbuf_local.start + t;"),
    ("writeback_via_local_range", "int64_t bi = bstart[k] + pc->gbuf_world_in_bucket.start + t;",
     "int64_t bi = bstart[k] + pc->gbuf_local.start + t;"),
    ("master_drops_piece_offset", "int64_t mi = pstart[p] + pc->param.start + t;",
     "int64_t mi = pstart[p] + t;"),
    ("writeback_drops_bucket_base", "int64_t bi = bstart[k] + pc->gbuf_world_in_bucket.start + t;",
     "int64_t bi = pc->gbuf_world_in_bucket.start + t;"),
    ("rank_range_shifted", "out->start = b_start + (int64_t)r * S;",
     "out->start = b_start + (int64_t)r * S + (r > 0);"),
    ("pad_ignores_D", "int64_t unit = (int64_t)D * (int64_t)pad_unit;", "int64_t unit = (int64_t)pad_unit;"),
    ("bucket_closes_late", "if (bucket_elems > 0 && open_count >= bucket_elems) {",
     "if (bucket_elems > 0 && open_count > bucket_elems) {"),
    ("local_range_from_bucket", "pc.gbuf_local = orc_normalize(pc.gbuf_world, x - mine.start);",
     "pc.gbuf_local = orc_normalize(pc.gbuf_world, x - bucket_start[k]);"),
    ("no_gather", "if (gather) {", "if (0) {"),
    ("allreduce_skips_own_rank",
     "for (int32_t q = 0; q < D; ++q) {\n                        if (grad_type == ORC_GRAD_F32)",
     "for (int32_t q = 0; q < D; ++q) {\n                        if (q == r) continue;\n"
     "                        if (grad_type == ORC_GRAD_F32)"),
    ("allreduce_truncates_bf16", "((uint16_t *)grads[q])[i - w0] = orc_f32_to_bf16(reduced);",
     "((uint16_t *)grads[q])[i - w0] = (uint16_t)(orc_f32_to_bits(reduced) >> 16);"),
    ("allreduce_via_bucket_range", "float reduced = shard[pc->gbuf_local.start + t];",
     "float reduced = shard[pc->gbuf_world_in_bucket.start + t];"),
    ("round_grad_ignored", "if (round_grad)\n                        g = orc_round_to_grad_type(g, grad_type);",
     "if (0)\n                        g = orc_round_to_grad_type(g, grad_type);"),
    ("round_grad_norm_unrounded",
     "if (round_grad)\n                r = orc_round_to_grad_type(r, grad_type);\n            double g",
     "if (0)\n                r = orc_round_to_grad_type(r, grad_type);\n            double g"),
    ("round_grad_truncates",
     "return grad_type == ORC_GRAD_F32 ? g : orc_bf16_to_f32(orc_f32_to_bf16(g));",
     "return grad_type == ORC_GRAD_F32 ? g : orc_bits_to_f32(orc_f32_to_bits(g) & 0xffff0000u);"),
    ("clip_not_applied", "float gc = g * clip_coef;", "float gc = g;"),
    ("norm_not_squared", "sum += g * g;", "sum += g < 0 ? -g : g;"),
    ("clip_no_sqrt", "double norm = sqrt(norm_sq);", "double norm = norm_sq;"),
    ("clip_no_upper_bound", "if (coef > 1.0)", "if (coef > 2.0)"),
    ("clip_eps_dropped", "double coef = (double)max_norm / (norm + 1e-6);",
     "double coef = (double)max_norm / norm;"),
    ("bf16_truncates", "if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))", "if (0)"),
    ("bf16_ties_away", "if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))",
     "if (lower >= 0x8000u)"),
    ("nonfinite_misses_nan", "if (isinf(r) || isnan(r))\n                ++count;",
     "if (isinf(r))\n                ++count;"),
    ("nonfinite_ignores_rounding",
     "r = orc_round_to_grad_type(r, grad_type);\n            if (isinf(r) || isnan(r))",
     "(void)0;\n            if (isinf(r) || isnan(r))"),
    ("nonfinite_counts_replicas", "if (isinf(r) || isnan(r))\n                ++count;",
     "for (int32_t q = 0; q < D; ++q) {\n                float x = orc_grad(grads, grad_type, q, i - w0);\n"
     "                if (isinf(x) || isnan(x))\n                    ++count;\n            }"),
    ("nonfinite_counts_past_piece_end",
     "int64_t i_hi = orc_min(pieces[pi].gbuf_world.end, w1);\n        for (int64_t i = i_lo; i < i_hi; ++i) {\n"
     "            float r = orc_reduce_element(grads, grad_type, D, instances, grad_scale, i - w0);\n"
     "            if (round_grad)\n                r = orc_round_to_grad_type(r, grad_type);\n            if (isinf",
     "int64_t i_hi = orc_min(pieces[pi].gbuf_world.end + 1, w1);\n        for (int64_t i = i_lo; i < i_hi; ++i) {\n"
     "            float r = orc_reduce_element(grads, grad_type, D, instances, grad_scale, i - w0);\n"
     "            if (round_grad)\n                r = orc_round_to_grad_type(r, grad_type);\n            if (isinf"),
    ("f16_widen_bias", "return orc_bits_to_f32(sign | ((e - 15u + 127u) << 23) | (frac << 13));",
     "return orc_bits_to_f32(sign | ((e - 14u + 127u) << 23) | (frac << 13));"),
    ("f16_widen_flushes_subnormals", "float v = (float)frac * 0x1p-24f;", "float v = 0.0f;"),
    ("f16_narrow_truncates", "double n = rint(ldexp(ax, 10 - ex));",
     "double n = floor(ldexp(ax, 10 - ex));"),
    ("f16_narrow_flushes_subnormals", "bits = (uint32_t)n; /* subnormal (ex == -14) */",
     "bits = 0u;"),
    ("f16_grads_read_as_bf16",
     "if (grad_type == ORC_GRAD_F16)\n        return orc_f16_to_f32(((const uint16_t *)grads[r])[idx]);",
     "if (0)\n        return orc_f16_to_f32(((const uint16_t *)grads[r])[idx]);"),
    ("f16_params_written_as_bf16", "uint16_t updated = param_is_f16 ? orc_f32_to_f16(",
     "uint16_t updated = 0 ? orc_f32_to_f16("),
    ("f16_round_grad_as_bf16", "if (grad_type == ORC_GRAD_F16)\n        return orc_f16_to_f32(orc_f32_to_f16(g));",
     "if (0)\n        return orc_f16_to_f32(orc_f32_to_f16(g));"),
    ("f16_allreduce_as_bf16", "else if (grad_type == ORC_GRAD_F16)\n                            ((uint16_t *)grads[q])[i - w0] = orc_f32_to_f16(reduced);",
     "else if (0)\n                            ((uint16_t *)grads[q])[i - w0] = orc_f32_to_f16(reduced);"),
]

RUNNER = r"""
import sys, traceback
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import oracle, pins
lib = oracle.load({path!r})
failed = []
for pin in pins.ALL_PINS:
    try:
        pin(lib)
    except BaseException as e:
        failed.append(pin.__name__)
        if {first_only!r}:
            break  # a mutant is caught by its first failing pin
print("FAILED_PINS", ",".join(failed))
sys.exit(1 if failed else 0)
"""


def _run_mutant(name, old, new, workdir):
    """Compile the oracle with one planted mistake and run the pins on it in
    a subprocess; returns (site found once, caught, output)."""
    with open(os.path.join(ROOT, "oracle", "dopt_oracle.c")) as f:
        src = f.read()
    if src.count(old) != 1:
        return False, False, f"mutation site for {name} not found exactly once"
    mutated = os.path.join(workdir, f"{name}.c")
    with open(mutated, "w") as f:
        f.write(src.replace(old, new))
    so = os.path.join(workdir, f"lib{name}.so")
    oracle._compile(mutated, so)
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), path=so, first_only=True)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                         timeout=600)
    return True, res.returncode != 0, res.stdout + res.stderr


@pytest.fixture(scope="module")
def mutant_results(tmp_path_factory):
    """Every mutant compiled and run at once (subprocesses in parallel: each
    is independent, and one that crashes takes only itself down)."""
    from concurrent.futures import ThreadPoolExecutor

    workdir = str(tmp_path_factory.mktemp("mutants"))
    workers = max(1, min(len(MUTANTS), os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        futures = {m[0]: ex.submit(_run_mutant, *m, workdir) for m in MUTANTS}
    return {name: f.result() for name, f in futures.items()}


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_mutant_is_caught(name, mutant_results):
    found, caught, output = mutant_results[name]
    assert found, output
    assert caught, f"mutant {name} passed every pin:\n{output}"


def test_runner_passes_unmutated_oracle():
    """Control: the same runner on the unmodified oracle reports no failure."""
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), path=oracle.build(),
                         first_only=False)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                         timeout=600)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "FAILED_PINS \n" in res.stdout or res.stdout.strip() == "FAILED_PINS"
