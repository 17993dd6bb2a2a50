"""Plants plausible mistakes into copies of the oracle (on the CPU) and
checks that at least one pin catches each.  This is evidence that the pins
constrain every part of the oracle: the total order, the causal bound, the
forced blocks, the tie-break, the output layout and the table expansion."""
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
from tests import oracle_pin_checks as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "bsa_oracle.c")

# (name, original text, mutated text)
MUTANTS = [
    ("zero_sign_ignored",
     "if (a.value == 0.0 && a.negative != b.negative) return a.negative ? -1 : 1;", ""),
    ("nan_sign_flipped",
     "if (a.is_nan) return a.negative ? -1 : 1;", "if (a.is_nan) return a.negative ? 1 : -1;"),
    ("negative_nan_payload_order",
     "if (a.negative) return a_smaller ? 1 : -1;", "if (a.negative) return a_smaller ? -1 : 1;"),
    ("page_rounding",
     "(len + ORACLE_PAGE_SIZE - 1) / ORACLE_PAGE_SIZE", "(len + ORACLE_PAGE_SIZE) / ORACLE_PAGE_SIZE"),
    ("causal_len_off_by_one",
     "int64_t causal_len = pos + 1 > 0 ? pos + 1 : 0;\n            out[req * dql + q]",
     "int64_t causal_len = pos > 0 ? pos : 0;\n            out[req * dql + q]"),
    ("varlen_position",
     "int64_t pos = (int64_t)prefix_lens[i] + (row - cu_seqlens_q[i]);",
     "int64_t pos = (int64_t)prefix_lens[i] + (row - cu_seqlens_q[i]) - 1;"),
    ("local_window_short",
     "(b >= v - num_local)", "(b > v - num_local)"),
    ("init_window_long",
     "(b < num_init)", "(b <= num_init)"),
    ("tie_break_higher_id",
     "return (a->id > b->id) - (a->id < b->id);", "return (a->id < b->id) - (a->id > b->id);"),
    ("descending_output",
     "return (a > b) - (a < b);", "return (a < b) - (a > b);"),
    ("tail_zero_not_minus_one",
     "dst[i] = i < n ? chosen[i] : -1;", "dst[i] = i < n ? chosen[i] : 0;"),
    ("forced_not_first",
     "if (a->forced != b->forced) return a->forced ? -1 : 1;", ""),
    ("order_reversed",
     "if (c != 0) return -c;", "if (c != 0) return c;"),
    ("table_page_bound_inclusive",
     "(int64_t)p * ORACLE_SUB_PAGE < causal_len", "(int64_t)p * ORACLE_SUB_PAGE <= causal_len"),
    ("table_ctx_full_blocks",
     "ctx += tokens < ORACLE_PAGE_SIZE ? tokens : ORACLE_PAGE_SIZE;", "ctx += ORACLE_PAGE_SIZE;"),
    ("table_accepts_causal_edge",
     "b >= num_blocks ||", "b > num_blocks ||"),
    ("table_keeps_duplicates",
     "if (!dup) blocks[n++] = b;", "(void)dup; blocks[n++] = b;"),
    ("table_phys_scale",
     "bt[j * ORACLE_PAGES_PER_BLOCK + p] = phys * ORACLE_PAGES_PER_BLOCK + p;",
     "bt[j * ORACLE_PAGES_PER_BLOCK + p] = phys + p;"),
    ("table_unsorted",
     "qsort(blocks, (size_t)n, sizeof(int32_t), int32_ascending);", ""),
    ("table_row_mapping",
     "int64_t local_q = r % dql;", "int64_t local_q = dql - 1 - r % dql;"),
    # mistakes inside the fused composition (select, then table)
    ("fused_strides_swapped",
     "T, H, M, token_stride, head_stride, nvp, K,", "T, H, M, head_stride, token_stride, nvp, K,"),
    ("fused_init_local_swapped",
     "num_init, num_local, out_idx);", "num_local, num_init, out_idx);"),
    ("fused_reads_capacity",
     "T, H, M, token_stride, head_stride, nvp, K,", "T, H, head_stride, token_stride, head_stride, nvp, K,"),
    ("fused_table_dql_one",
     "B, MB, seq_lens,\n                                             dql, sparse_bt",
     "B, MB, seq_lens,\n                                             1, sparse_bt"),
    ("fused_table_from_page_counts",
     "rc = oracle_build_sparse_block_table(out_idx, T, H, K, block_table, B, MB, seq_lens,",
     "rc = oracle_build_sparse_block_table(out_idx, T, H, K, block_table, B, MB, nvp,"),
    # mistakes in the index scores
    ("score_logical_block_as_physical",
     "const int64_t phys = b < MB ? block_table[req * MB + b] : -1;",
     "const int64_t phys = b < MB ? b : -1;"),
    ("score_head_ignored",
     "const uint16_t* qv = q + (t * H + h) * D;", "const uint16_t* qv = q + (t * H) * D;"),
    ("score_row_position",
     "const int64_t pos = (int64_t)seq_lens[req] - dql + lq;",
     "const int64_t pos = (int64_t)seq_lens[req] - dql + lq + 1;"),
    ("score_missing_key_zero",
     "row[b] = -INFINITY;", "row[b] = 0.0;"),
    ("score_key_transposed",
     "decode_bits(k[phys * D + d], 8, 7)", "decode_bits(k[phys + d * NB], 8, 7)"),
    # mistakes in the sparse decode attention
    ("attn_scale_dropped",
     "s[j] = scale * dot;", "s[j] = dot;"),
    ("attn_key_slot_reversed",
     "k_cache + ((page * ORACLE_SUB_PAGE + j % ORACLE_SUB_PAGE) * H + h) * D;",
     "k_cache + ((page * ORACLE_SUB_PAGE + 15 - j % ORACLE_SUB_PAGE) * H + h) * D;"),
    ("attn_value_head_ignored",
     "v_cache + ((page * ORACLE_SUB_PAGE + j % ORACLE_SUB_PAGE) * H + h) * D;",
     "v_cache + ((page * ORACLE_SUB_PAGE + j % ORACLE_SUB_PAGE) * H) * D;"),
    ("attn_last_token_dropped",
     "if (ctx > width * ORACLE_SUB_PAGE) ctx = width * ORACLE_SUB_PAGE;",
     "if (ctx > width * ORACLE_SUB_PAGE) ctx = width * ORACLE_SUB_PAGE;\n            ctx -= ctx > 0;"),
]


def _build_mutant(tmp, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutant {name}: pattern must occur exactly once"
    path = os.path.join(tmp, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    so = os.path.join(tmp, f"lib{name}.so")
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-w", "-fPIC", "-shared", "-o", so, path, "-lm"])
    return oracle.load_library(so)


@pytest.fixture(scope="module")
def tmpdir_mod():
    d = tempfile.mkdtemp(prefix="bsa_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmpdir_mod, name, old, new):
    lib = _build_mutant(tmpdir_mod, name, old, new)
    # the pins of the mutated part first (any order would do; this one is faster)
    part = {"attn": "attention", "score": "index_scores", "fused": "fused",
            "table": "table"}.get(name.split("_")[0], "")
    order = sorted(pins.ALL_CHECKS, key=lambda c: part == "" or part not in c.__name__)
    for check in order:
        try:
            check(lib=lib)
        except AssertionError:
            return        # caught by this pin
    raise AssertionError(f"no pin catches mutant {name}")
