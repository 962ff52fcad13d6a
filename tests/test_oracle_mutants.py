"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each one.

Each mutant is one textual edit — a dropped term, a wrong sign, a transposed
index, an off-by-one. Edits of oracle/pkv_oracle.c are compiled to a
temporary library and run under tests/test_oracle_pins.py (the oracle loader
takes the library path from PKV_ORACLE_LIB); edits of oracle/blockmgr.py are
written to a temporary file and run under tests/test_blockmgr_pins.py (which
loads the file named by PKV_ORACLE_BLOCKMGR). A mutant that passes every pin
would mean the pins cannot tell that mistake from the pages' rules.
"""
import concurrent.futures as cf
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pkv_oracle.c")
BM_SRC = os.path.join(ROOT, "oracle", "blockmgr.py")

MUTANTS = {
    "drop_normalisation": ("for (int d = 0; d < dim; ++d) o[d] /= sum;", ""),
    "max_subtraction_sign": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "drop_scale": ("s[j] = scale * dot;", "s[j] = dot;"),
    "layout_head_before_kv": ("    i = i * 2 + kv;\n    i = i * g->num_heads + h;",
                              "    i = i * g->num_heads + h;\n    i = i * 2 + kv;"),
    "layout_token_dim_swapped": ("    i = i * g->block_size + t;\n    return i * g->head_dim + d;",
                                 "    i = i * g->head_dim + d;\n    return i * g->block_size + t;"),
    "gather_last_block_wrong": ("pool[elem(g, table[full], layer, kv, head, t, d)]",
                                "pool[elem(g, table[0], layer, kv, head, t, d)]"),
    "slot_forgets_block_scale": ("return (int64_t)table[pos / block_size] * block_size + pos % block_size;",
                                 "return (int64_t)table[pos / block_size] + pos % block_size;"),
    "append_v_gets_k": ("pool[elem(g, b, layer, 1, h, t, d)] = v[src];",
                        "pool[elem(g, b, layer, 1, h, t, d)] = k[src];"),
    "half_encode_truncates": ("double r = rint(ldexp(a, 10 - ue));", "double r = floor(ldexp(a, 10 - ue));"),
    "half_decode_subnormal_scale": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "causal_excludes_self": ("pkvo_attend(qd, K, V, pos + 1, D, scale, o);", "pkvo_attend(qd, K, V, pos, D, scale, o);"),
    "prefill_position_shift": ("pos = n - qlen + i;", "pos = n - qlen + i - (i > 0);"),
    "merge_unweighted_sum": ("L += w * l[p];", "L += l[p];"),
    "bytes_drop_kv_factor": ("return 2LL * g->num_layers * g->num_heads * g->head_dim * 2;",
                             "return 1LL * g->num_layers * g->num_heads * g->head_dim * 2;"),
    "ceil_becomes_floor": ("return (tokens + block_size - 1) / block_size;", "return tokens / block_size;"),
    "partial_exp_drops_scale": ("double p = exp(scale * dot - m);", "double p = exp(dot - m);"),
    "gqa_heads_interleaved": ("return h / (pkvo_q_heads(g) / g->num_heads);", "return h % g->num_heads;"),
    "i8_reads_scale_of_token0": ("memcpy(&scale, tile + (int64_t)g->block_size * g->head_dim + 4LL * t, 4);\n    return",
                                 "memcpy(&scale, tile + (int64_t)g->block_size * g->head_dim, 4);\n    return"),
    "i8_amax_signed": ("float a = (float)fabs(pkvo_half_to_double(x[i]));",
                       "float a = (float)pkvo_half_to_double(x[i]);"),
    "i8_code_truncates": ("c = (int)rintf(qv);", "c = (int)qv;"),
    "copy_blocks_direction": ("memmove((char*)pool + pairs[2 * i + 1] * bb, (const char*)pool + pairs[2 * i] * bb, (size_t)bb);",
                              "memmove((char*)pool + pairs[2 * i] * bb, (const char*)pool + pairs[2 * i + 1] * bb, (size_t)bb);"),
    "swap_in_ignores_host_offset": ("memcpy((char*)pool + blocks[i] * bb, (const char*)host + i * bb, (size_t)bb);",
                                    "memcpy((char*)pool + blocks[i] * bb, (const char*)host, (size_t)bb);"),
    "fnv_prime_off_by_two": ("h *= 1099511628211ULL;", "h *= 1099511628213ULL;"),
    "hash_chain_restarts": ("for (int k = 0; k < 8; ++k) buf[k] = (uint8_t)(h >> (8 * k));",
                            "for (int k = 0; k < 8; ++k) buf[k] = 0;"),
    "i8_tile_head_before_kv": ("((b * g->num_layers + l) * 2 + kv) * g->num_heads + h;",
                               "((b * g->num_layers + l) * g->num_heads + h) * 2 + kv;"),
    "gqa_q_stride_uses_kv_heads": ("    const int H = pkvo_q_heads(g), D = g->head_dim;\n    #pragma omp parallel for collapse(2) schedule(dynamic)\n    for (int r = 0; r < B; ++r)\n        for (int h = 0; h < H; ++h) {\n            int64_t n = ctx_lens[r];\n            double* K",
                                   "    const int H = g->num_heads, D = g->head_dim;\n    #pragma omp parallel for collapse(2) schedule(dynamic)\n    for (int r = 0; r < B; ++r)\n        for (int h = 0; h < H; ++h) {\n            int64_t n = ctx_lens[r];\n            double* K"),
}


# mistakes in the block manager's restatement (oracle/blockmgr.py)
BM_MUTANTS = {
    # the reading that made a fork at 47 tokens unable to take its 48th: look at position len, not len - 1
    "cow_looks_past_last_position": ("range((n - num_new) // self.block_size, (n - 1) // self.block_size + 1)",
                                     "range(n // self.block_size, n // self.block_size + 1)"),
    "cow_off_by_one_last_block": ("(n - 1) // self.block_size + 1) if num_new", "(n - 1) // self.block_size) if num_new"),
    "cow_copies_last_shared_not_first": ("i = shared[0]", "i = shared[-1]"),
    "cow_keeps_old_reference": ("        old = t[i]\n        self.ref[old] -= 1\n", "        old = t[i]\n"),
    "evict_most_recently_used_first": ("cand = sorted((e[1], -e[2], e[0], h)", "cand = sorted((-e[1], -e[2], e[0], h)"),
    "evict_shallow_first": ("cand = sorted((e[1], -e[2], e[0], h)", "cand = sorted((e[1], e[2], e[0], h)"),
    "evict_referenced_entries": ("if self.ref[e[0]] == 1)", "if self.ref[e[0]] >= 1)"),
    "attach_does_not_refresh_use": ("            e[1] = self.clock\n            self.ref[e[0]] += 1",
                                    "            self.ref[e[0]] += 1"),
    "grow_pops_from_front": ("        for _ in range(max(need, 0)):\n            b = self.free.pop()",
                             "        for _ in range(max(need, 0)):\n            b = self.free.pop(0)"),
    "fork_skips_last_block": ("        for b in self.tables[src]:\n            self.ref[b] += 1\n        self.tables[dst] = list(self.tables[src])",
                              "        for b in self.tables[src][:-1]:\n            self.ref[b] += 1\n        self.tables[dst] = list(self.tables[src])"),
    "share_prefix_allows_partial_block": ("n_blocks * self.block_size > self.lens[src]",
                                          "(n_blocks - 1) * self.block_size > self.lens[src]"),
    "build_step_allows_shared_write": ("if self.ref[b] != 1:", "if self.ref[b] > 2:"),
    "match_skips_a_miss": ("            if int(h) not in self.cache:\n                break",
                           "            if int(h) not in self.cache:\n                continue"),
    "swap_in_ignores_partial_block": ("need = self.blocks_needed(self.lens[seq])", "need = self.lens[seq] // self.block_size"),
}


def _run_bm_mutant(name, tmp):
    find, repl = BM_MUTANTS[name]
    src = open(BM_SRC).read()
    assert src.count(find) == 1, f"mutant {name}: pattern must occur exactly once"
    path = os.path.join(tmp, f"bm_{name}.py")
    with open(path, "w") as f:
        f.write(src.replace(find, repl))
    env = dict(os.environ, PKV_ORACLE_BLOCKMGR=path)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_blockmgr_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode, r.stdout[-400:]


def _run_mutant(name, tmp):
    find, repl = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(find) == 1, f"mutant {name}: pattern must occur exactly once"
    path_c = os.path.join(tmp, f"{name}.c")
    path_so = os.path.join(tmp, f"lib{name}.so")
    with open(path_c, "w") as f:
        f.write(src.replace(find, repl))
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", path_c,
                    "-o", path_so, "-lm"], check=True)
    env = dict(os.environ, PKV_ORACLE_LIB=path_so, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode, r.stdout[-400:]


def test_every_planted_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
            results = list(ex.map(lambda n: _run_mutant(n, tmp), sorted(MUTANTS)))
    survivors = [(n, out) for n, rc, out in results if rc == 0]
    assert not survivors, f"mutants not caught by any pin: {survivors}"
    # a return code of 1 means tests ran and failed (not a crash of the harness)
    assert all(rc in (1, -11, -6) or rc > 1 for _, rc, _ in results)


def test_every_planted_block_manager_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
            results = list(ex.map(lambda n: _run_bm_mutant(n, tmp), sorted(BM_MUTANTS)))
    survivors = [(n, out) for n, rc, out in results if rc == 0]
    assert not survivors, f"mutants not caught by any pin: {survivors}"
    assert all(rc == 1 for _, rc, _ in results), results


def test_unmutated_block_manager_passes_its_pins_when_loaded_from_a_file():
    # the harness itself: the original file, loaded the way the mutants are, passes
    env = dict(os.environ, PKV_ORACLE_BLOCKMGR=BM_SRC)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_blockmgr_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-800:]
