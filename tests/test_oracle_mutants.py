"""The oracle's pins catch planted mistakes (CPU only).

Each case below plants one plausible slip in a copy of the oracle's C source: an off-by-one
causal mask, a wrong KV group, page or request index, a reversed tie rule, a dropped forced
block, a dropped softmax normaliser or max shift, a wrong merge weight, a wrong bucket
offset, a wrong bf16 rounding, an ignored unit list, rows skipped by the thread split. The
copy is compiled on its own and the whole pin suite
(``test_oracle_pins.py``) runs against it in a child process; every copy must fail at least
one pin. An unmodified copy run the same way must pass, so a broken harness cannot make
every slip look caught. Mistakes are planted only in these temporary copies, never in the
oracle itself, and nothing here touches a GPU.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "msa_oracle.c")

# (slip, text of the oracle it replaces -- must occur exactly once, replacement)
MUTANTS = [
    # stage 1: block scores
    ("score: causal mask off by one",
     "          if (pos > q_pos) break;\n          const uint16_t* k = c->k_idx",
     "          if (pos >= q_pos) break;\n          const uint16_t* k = c->k_idx"),
    ("score: key index of group 0",
     "((page * MSA_BLOCK + tau) * c->Hkv + g) * c->Di",
     "((page * MSA_BLOCK + tau) * c->Hkv + 0) * c->Di"),
    ("score: query index of group 0",
     "c->q_idx + (r * c->Hkv + g) * c->Di", "c->q_idx + (r * c->Hkv) * c->Di"),
    ("score: last token instead of the block max",
     "if (acc > best) best = acc;", "best = acc;"),
    ("score: local block left unscored",
     "(int64_t)j <= q_pos / MSA_BLOCK", "(int64_t)j < q_pos / MSA_BLOCK"),
    ("score: page table row of request 0",
     "int64_t page = c->page_table[b * c->max_blocks + j];\n        for (int tau",
     "int64_t page = c->page_table[j];\n        for (int tau"),
    ("score: every row at the last position",
     "int64_t q_pos = (int64_t)c->seq_lens[b] - c->N + i;",
     "int64_t q_pos = (int64_t)c->seq_lens[b] - 1;"),
    ("score: key channels reversed",
     "acc += bf16_to_f32(q[d]) * bf16_to_f32(k[d]);",
     "acc += bf16_to_f32(q[d]) * bf16_to_f32(k[c->Di - 1 - d]);"),
    # stage 1: top-k
    ("topk: ties to the higher id",
     "return (x->id > y->id) - (x->id < y->id);", "return (x->id < y->id) - (x->id > y->id);"),
    ("topk: local block not forced", "if (local > 0) kept[nk++] = (int)local;", ""),
    ("topk: sink block not forced", "kept[nk++] = 0;\n", ""),
    ("topk: lowest scores kept",
     "if (x->s > y->s) return -1;\n  if (x->s < y->s) return 1;",
     "if (x->s < y->s) return -1;\n  if (x->s > y->s) return 1;"),
    ("topk: ids left in score order", "qsort(kept, (size_t)nk, sizeof(int), int_cmp);", ""),
    ("topk: block 1 never a candidate",
     "for (int j = 1; j < local; ++j) { cands", "for (int j = 2; j < local; ++j) { cands"),
    ("topk: selected score read by slot",
     "i < nk ? s[kept[i]] : -INFINITY;", "i < nk ? s[i] : -INFINITY;"),
    # sparse page table
    ("page table: virtual page without the group",
     "(int32_t)(p * MSA_BLOCK * Hkv + g)", "(int32_t)(p * MSA_BLOCK * Hkv)"),
    ("page table: local block length off by one",
     "(q_pos % MSA_BLOCK) + 1 : MSA_BLOCK", "(q_pos % MSA_BLOCK) : MSA_BLOCK"),
    ("page table: every row at the last position",
     "int64_t q_pos = (int64_t)seq_lens[b] - N + (r % N);",
     "int64_t q_pos = (int64_t)seq_lens[b] - 1;"),
    ("page table: page row of request 0",
     "int64_t p = page_table[b * max_blocks + j];", "int64_t p = page_table[j];"),
    # softmax attention core
    ("attention: half the max shift", "double p = exp(s_buf[i] - m);",
     "double p = exp(s_buf[i] - m / 2);"),
    ("attention: lse without the max", "*lse = m + log(l);", "*lse = log(l);"),
    ("attention: no normalisation", "for (int d = 0; d < D; ++d) o[d] /= l;", ""),
    ("attention: scores against values",
     "(double)bf16_to_f32(q[d]) * (double)bf16_to_f32(keys[i][d]);",
     "(double)bf16_to_f32(q[d]) * (double)bf16_to_f32(vals[i][d]);"),
    # decode (logical and through the strided view)
    ("decode: head to group by modulo",
     "  int g = h / (c->Hq / c->Hkv);\n  int64_t b = r / c->N;",
     "  int g = h % c->Hkv;\n  int64_t b = r / c->N;"),
    ("decode: causal mask off by one",
     "      if (pos > q_pos) break;\n      int64_t off = ((page",
     "      if (pos >= q_pos) break;\n      int64_t off = ((page"),
    ("decode: every row at the last position",
     "int64_t q_pos = (int64_t)c->seq_lens[b] - c->N + (r % c->N);",
     "int64_t q_pos = (int64_t)c->seq_lens[b] - 1;"),
    ("decode: K/V of group 0",
     "int64_t off = ((page * MSA_BLOCK + tau) * c->Hkv + g) * c->D;",
     "int64_t off = ((page * MSA_BLOCK + tau) * c->Hkv) * c->D;"),
    ("decode: page table row of request 0",
     "int64_t page = c->page_table[b * c->max_blocks + j];\n    for (int tau",
     "int64_t page = c->page_table[j];\n    for (int tau"),
    ("decode: selection of group 0",
     "const int32_t* ids = c->block_ids + (r * c->Hkv + g) * c->topk;",
     "const int32_t* ids = c->block_ids + (r * c->Hkv) * c->topk;"),
    ("strided view: token stride without the groups",
     "(t % MSA_BLOCK) * (int64_t)c->Hkv * c->D;", "(t % MSA_BLOCK) * (int64_t)c->D;"),
    ("strided view: head to group by modulo",
     "int64_t f = r * c->Hkv + h / (c->Hq / c->Hkv);", "int64_t f = r * c->Hkv + h % c->Hkv;"),
    # prefill, block partials, merge, bucketing
    ("prefill: head to group by modulo",
     "  int g = h / (c->Hq / c->Hkv);\n  int64_t q_pos = c->S",
     "  int g = h % c->Hkv;\n  int64_t q_pos = c->S"),
    ("prefill: causal mask off by one",
     "if (pos > q_pos || pos >= c->S) break;", "if (pos >= q_pos || pos >= c->S) break;"),
    ("prefill: chunk starting at position 0",
     "int64_t q_pos = c->S - c->T + t;", "int64_t q_pos = t;"),
    ("prefill: selection of group 0",
     "const int32_t* ids = c->block_ids + (t * c->Hkv + g) * c->topk;",
     "const int32_t* ids = c->block_ids + (t * c->Hkv) * c->topk;"),
    ("block partial: no causal mask",
     "if (pos > q_pos || pos >= S_kv) break;", "if (pos >= S_kv) break;"),
    ("block partial: head to group by modulo",
     "  int g = h / (Hq / Hkv);\n  int64_t q_pos = S_kv", "  int g = h % Hkv;\n  int64_t q_pos = S_kv"),
    ("merge: weights not normalised",
     "double w = exp((double)lse_parts[i] - out_lse);", "double w = exp((double)lse_parts[i] - m);"),
    ("merge: lse is the largest partial lse", "*lse = out_lse;", "*lse = m;"),
    ("merge: last partial left out of the normaliser",
     "for (int i = 0; i < n; ++i) total += exp", "for (int i = 0; i + 1 < n; ++i) total += exp"),
    ("buckets: entry without its slot",
     "= (int32_t)(t * topk + i);", "= (int32_t)(t * topk);"),
    ("buckets: every group's lists from offset 0", "base += off[nblk];", ""),
    ("buckets: last block never counted",
     "if (j >= 0 && j < nblk) off[j + 1] += 1;", "if (j >= 0 && j < nblk - 1) off[j + 1] += 1;"),
    # unit and row lists (the sampled form of the full-size comparisons), thread split
    ("decode: unit list ignored",
     "  dec_ctx* c = (dec_ctx*)p;\n  int64_t u = c->units ? c->units[slot] : slot;",
     "  dec_ctx* c = (dec_ctx*)p;\n  int64_t u = slot;"),
    ("strided view: unit list ignored",
     "  flat_ctx* c = (flat_ctx*)p;\n  int64_t u = c->units ? c->units[slot] : slot;",
     "  flat_ctx* c = (flat_ctx*)p;\n  int64_t u = slot;"),
    ("prefill: unit list ignored",
     "  pre_ctx* c = (pre_ctx*)p;\n  int64_t u = c->units ? c->units[slot] : slot;",
     "  pre_ctx* c = (pre_ctx*)p;\n  int64_t u = slot;"),
    ("score: row list ignored",
     "int64_t r = c->rows ? c->rows[slot] : slot;", "int64_t r = slot;"),
    ("threads: rows skipped", "i += a->nthreads) a->fn", "i += a->nthreads + 1) a->fn"),
    # padding, empty rows and other edge cases
    ("attention: a row with no visible key gets lse 0",
     "if (n == 0) { *lse = -INFINITY; return; }", "if (n == 0) { *lse = 0.0; return; }"),
    ("merge: only -inf partials give a NaN lse",
     "if (n == 0 || m == -INFINITY) { *lse = -INFINITY; return 0; }",
     "if (n == 0) { *lse = -INFINITY; return 0; }"),
    ("attention: scores accumulated in float",
     "    double acc = 0.0;\n    for (int d = 0; d < D; ++d) acc += (double)",
     "    float acc = 0.0f;\n    for (int d = 0; d < D; ++d) acc += (double)"),
    ("score: blocks past the query score 0",
     "      out[j] = best;", "      out[j] = best == -INFINITY ? 0.0f : best;"),
    ("topk: block 0 kept twice when it is the local block",
     "if (local > 0) kept[nk++] = (int)local;", "kept[nk++] = (int)local;"),
    ("topk: padding id 0", "ids[i] = i < nk ? kept[i] : -1;", "ids[i] = i < nk ? kept[i] : 0;"),
    ("topk: padding score 0", "i < nk ? s[kept[i]] : -INFINITY;", "i < nk ? s[kept[i]] : 0.0f;"),
    ("page table: padding on page 0",
     "if (j < 0) { flat_page_table[f * topk + i] = -1; continue; }",
     "if (j < 0) { flat_page_table[f * topk + i] = 0; continue; }"),
    ("bf16: NaN rounded to infinity", "if (isnan(x)) return 0x7fc0;", "if (isnan(x)) return 0x7f80;"),
    ("bf16: negative zero loses its sign",
     "if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;", "if (x == 0.0) return 0x0000;"),
    # bf16 rounding
    ("bf16: truncation", "y = ldexp(nearbyint(ldexp(m, 8)), e - 8);",
     "y = ldexp(trunc(ldexp(m, 8)), e - 8);"),
    ("bf16: ties away from zero", "y = ldexp(nearbyint(ldexp(m, 8)), e - 8);",
     "y = ldexp(round(ldexp(m, 8)), e - 8);"),
    ("bf16: subnormal quantum doubled", "y = ldexp(nearbyint(ldexp(x, 133)), -133);",
     "y = ldexp(nearbyint(ldexp(x, 132)), -132);"),
]

# Run the pin suite with the oracle package loading the given library instead of its own.
_RUN_PINS = (
    "import sys\n"
    "import oracle\n"
    "lib = sys.argv[1]\n"
    "oracle.build = lambda force=False: lib\n"
    "import pytest\n"
    "sys.exit(pytest.main(['-x', '-q', '-p', 'no:cacheprovider', 'tests/test_oracle_pins.py']))\n")


def _pins_pass_with(source: str, workdir: str) -> bool:
    os.makedirs(workdir, exist_ok=True)
    src = os.path.join(workdir, "oracle_variant.c")
    lib = os.path.join(workdir, "liboracle_variant.so")
    with open(src, "w") as f:
        f.write(source)
    subprocess.run(oracle.gcc_command(src, lib), check=True, capture_output=True)
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-c", _RUN_PINS, lib], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    if r.returncode not in (0, 1):  # 1: a pin failed; anything else: the run itself broke
        raise RuntimeError(f"pin run ended with {r.returncode}:\n{r.stdout[-2000:]}{r.stderr[-2000:]}")
    return r.returncode == 0


def test_every_planted_mistake_fails_a_pin(tmp_path):
    with open(SRC) as f:
        original = f.read()
    for slip, old, _ in MUTANTS:
        assert original.count(old) == 1, f"{slip}: its text occurs {original.count(old)} times"

    jobs = [("unmodified copy", original)] + [(slip, original.replace(old, new))
                                             for slip, old, new in MUTANTS]
    workers = max(1, min(8, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        passed = dict(zip([name for name, _ in jobs],
                          ex.map(lambda ij: _pins_pass_with(ij[1][1], str(tmp_path / f"v{ij[0]}")),
                                 enumerate(jobs))))
    assert passed.pop("unmodified copy"), "the pins fail on an unmodified copy of the oracle"
    survivors = [slip for slip, ok in passed.items() if ok]
    assert not survivors, f"planted mistakes no pin catches: {survivors}"
