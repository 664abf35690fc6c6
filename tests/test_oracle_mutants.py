"""Planted mistakes in the oracle must each fail at least one pin (no GPU).

Every mutant below is a plausible slip in the oracle (a wrong index, a dropped
term, a transposed operand, a LIFO instead of a FIFO ...).  The test compiles a
copy of the oracle source with that one change and runs the pin suite against it;
the suite must fail.  The planted copies live in a temporary directory only.
"""
import concurrent.futures
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pkv_oracle.cpp")

MUTANTS = {
    "lifo_free_list": ("if (P.ref[p] == 0) P.free_fifo.push_back(p);", "if (P.ref[p] == 0) P.free_fifo.push_front(p);"),
    "cow_on_sole_owner": ("} else if (P.ref[s.table[l]] > 1) {", "} else if (P.ref[s.table[l]] >= 1) {"),
    "cow_keeps_old_owner": ("release_block(P, old);  // count", "(void)old;  // count"),
    "cow_pair_reversed": ("cow_pairs[2 * cows] = old;", "cow_pairs[2 * cows] = p;"),
    "offset_from_wrong_slot": ("slot_mapping[start[i] + k] = static_cast<int32_t>(s.table[l] * P.B + o);",
                               "slot_mapping[start[i] + k] = static_cast<int32_t>(s.table[l] * P.B + (P.B - 1 - o));"),
    "fork_forgets_length": ("c.len = it->second.len;", "c.len = 0;"),
    "fork_no_refcount": ("for (int32_t p : c.table) P.ref[p] += 1;", "for (int32_t p : c.table) (void)p;"),
    "gqa_head_interleaved": ("const int h = g * G + hh;", "const int h = hh * H_kv + g;"),
    "scale_dropped": ("z[t] = scale * acc;", "z[t] = acc;"),
    "scores_against_values": ("for (int i = 0; i < d; ++i) acc += qv[i] * K[t * d + i];",
                              "for (int i = 0; i < d; ++i) acc += qv[i] * V[t * d + i];"),
    "weights_keys": ("for (int i = 0; i < d; ++i) o[i] += w * V[t * d + i];",
                     "for (int i = 0; i < d; ++i) o[i] += w * K[t * d + i];"),
    "gather_wrong_block": ("int64_t p = tables[static_cast<int64_t>(s) * W + t / B];",
                           "int64_t p = tables[static_cast<int64_t>(s) * W + (t / B + 1) % ((len + B - 1) / B)];"),
    "half_exponent_bias": ("v = std::ldexp(1.0 + frac / 1024.0, expo - 15);", "v = std::ldexp(1.0 + frac / 1024.0, expo - 16);"),
    "frame_size_halved": ("char* frame = static_cast<char*>(host) + host_slots[i] * 2 * blk;",
                          "char* frame = static_cast<char*>(host) + host_slots[i] * blk;"),
    "block_bytes_no_heads": ("const size_t blk = static_cast<size_t>(L) * H_kv * B * d * elem_bytes(dtype);\n  for (int64_t i = 0; i < n; ++i) {\n    int32_t s = pairs",
                             "const size_t blk = static_cast<size_t>(L) * B * d * elem_bytes(dtype);\n  for (int64_t i = 0; i < n; ++i) {\n    int32_t s = pairs"),
    "write_skips_value": ("std::memcpy(static_cast<char*>(v_pool) + dst, static_cast<const char*>(v_new) + src, row);",
                          "(void)v_new;"),
    "softmax_not_normalised": ("double w = std::exp(z[t] - zmax) / denom;", "double w = std::exp(z[t] - zmax);"),
    "prefill_sees_one_less": ("const int64_t visible = P + qi + 1;", "const int64_t visible = P + qi;"),
    "prefill_forgets_history": ("const int64_t visible = P + qi + 1;", "const int64_t visible = qi + 1;"),
    "e4m3_bias_8": ("v = std::ldexp(1.0 + frac / 8.0, expo - 7);", "v = std::ldexp(1.0 + frac / 8.0, expo - 8);"),
    "e4m3_subnormal_step": ("v = std::ldexp(static_cast<double>(frac), -9);",
                            "v = std::ldexp(static_cast<double>(frac), -10);"),
    "e4m3_ties_upward": ("if (err < best_err || (err == best_err && (c & 1) == 0)) {", "if (err <= best_err) {"),
    "e4m3_no_448": ("for (int c = 0; c <= 0x7e; ++c) {", "for (int c = 0; c < 0x7e; ++c) {"),
    "quantise_by_product": ("const float kq = bf16_at(k_new, src + e) / k_scale;",
                            "const float kq = bf16_at(k_new, src + e) * k_scale;"),
    "key_scale_dropped": ("K[t * d + i] = k_scale * decode(k_pool, base + i, dtype);",
                          "K[t * d + i] = decode(k_pool, base + i, dtype);"),
    "swap_in_lifo": ("    allocate_block(P, &p);\n    s.table.push_back(p);",
                     "    p = P.free_fifo.back(); P.free_fifo.pop_back(); P.ref[p] = 1;\n    s.table.push_back(p);"),
}


def _run_mutant(name, old, new, tmp):
    src = open(SRC).read()
    # a slip in a line the two attention functions share is planted in both
    assert src.count(old) >= 1, f"mutant {name}: anchor not found"
    mdir = os.path.join(tmp, name)
    os.makedirs(mdir)
    cpp = os.path.join(mdir, "m.cpp")
    lib = os.path.join(mdir, "libm.so")
    open(cpp, "w").write(src.replace(old, new))
    subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread", cpp, "-o", lib], check=True)
    env = dict(os.environ, PKV_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode


def test_every_planted_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with concurrent.futures.ThreadPoolExecutor(max_workers=max(2, (os.cpu_count() or 2))) as ex:
            futs = [ex.submit(_run_mutant, n, o, w, tmp) for n, (o, w) in MUTANTS.items()]
            results = dict(f.result() for f in futs)
    survivors = [n for n, rc in results.items() if rc == 0]
    assert not survivors, f"pins did not catch: {survivors}"
