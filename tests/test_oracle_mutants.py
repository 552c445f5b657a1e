"""Planted mistakes in the oracle must fail at least one pin.

Each case copies kvx_oracle.c, plants one plausible mistake (a dropped term, a wrong index, a
transposed operand, a skipped check), builds the copy with the host compiler and runs every
pin against it.  The real oracle source is never modified.
"""
import json
import os
import shutil
import subprocess
import sys
import tempfile

import pytest

import oracle
from tests import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kvx_oracle.c")
HDR = os.path.join(os.path.dirname(oracle.__file__), "kvx_oracle.h")

MUTANTS = {
    "kv_swapped_in_buffer": ("(((int64_t)plane * n + token) * pool->kv_heads",
                             "(((int64_t)(plane ^ 1) * n + token) * pool->kv_heads"),
    "hnd_page_offset_off_by_one": ("* pool->page_size + off) * hb",
                                   "* pool->page_size + (off + 1) % pool->page_size) * hb"),
    "hnd_heads_and_offsets_transposed": ("((page * pool->kv_heads + head) * pool->page_size + off)",
                                         "((page * pool->page_size + off) * pool->kv_heads + head)"),
    "nhd_head_stride_dropped": ("return base + slot * pool->slot_stride + head * hb;",
                                "return base + slot * pool->slot_stride;"),
    "range_check_off_by_one": ("(int64_t)slots[i] >= pool->num_slots",
                               "(int64_t)slots[i] > pool->num_slots"),
    "negative_slot_accepted": ("slots[i] < 0 || (int64_t)slots[i] >= pool->num_slots",
                               "(int64_t)slots[i] >= pool->num_slots"),
    "permute_missing": ("memcpy(buf_vec(buf, src, p, seq_len, s, h), logical + ((int64_t)h * seq_len + s) * hb,",
                        "memcpy(buf_vec(buf, src, p, seq_len, s, h), logical + ((int64_t)s * H + h) * hb,"),
    "factor_two_dropped": ("return (int64_t)2 * num_layers", "return (int64_t)num_layers"),
    "runs_dst_break_dropped": (" &&\n           (int64_t)dst_idx[b] == (int64_t)dst_idx[b - 1] + 1)", ")"),
    "runs_request_break_dropped": ("const int64_t req_end = (q + 1 < n_reqs) ? req_start[q + 1] : n;",
                                   "const int64_t req_end = n;"),
    "runs_src_step_of_two": ("(int64_t)src_idx[b] == (int64_t)src_idx[b - 1] + 1 &&",
                             "(int64_t)src_idx[b] >= (int64_t)src_idx[b - 1] + 1 &&"),
    "runs_step_in_32_bits": ("(int64_t)src_idx[b] == (int64_t)src_idx[b - 1] + 1 &&",
                             "(uint32_t)src_idx[b] == (uint32_t)src_idx[b - 1] + 1u &&"),
    "batch_status_not_per_request": ("status[1 + q] = rc;", "status[1 + q] = 0;"),
    "batch_dup_pairs_missed": ("if (count[dst_slots[r->dst_off + i]] > 1) {",
                               "if (count[dst_slots[r->dst_off + i]] > 2) {"),
    "batch_dup_counts_refused_requests": ("const int counted = status[1 + q] == KVXO_OK && r->op != KVXO_OP_GATHER;",
                                          "const int counted = r->op != KVXO_OP_GATHER;"),
    "batch_dup_check_ignored": ("if (check_dup && dst) {", "if (0 && dst) {"),
    "layers_one_short": ("for (int32_t layer = 0; layer < stop; ++layer)\n    for (int32_t kv = 0; kv < ppl; ++kv)\n      for (int64_t i = 0; i < n; ++i)\n        for",
                         "for (int32_t layer = 0; layer + 1 < stop; ++layer)\n    for (int32_t kv = 0; kv < ppl; ++kv)\n      for (int64_t i = 0; i < n; ++i)\n        for"),
    "layers_v_plane_dropped": ("    for (int32_t kv = 0; kv < ppl; ++kv)\n      for (int64_t i = 0; i < n; ++i)\n        for",
                               "    for (int32_t kv = 0; kv < 1; ++kv)\n      for (int64_t i = 0; i < n; ++i)\n        for"),
    "tp_replicas_all_send": ("  if (p_tp > heads && p_rank % (p_tp / heads) != 0) return KVXO_OK; /* another replica sends */\n", ""),
    "tp_dst_offset_from_p_side": ("  *dst_head0 = lo - df;", "  *dst_head0 = lo - pf;"),
    "heads_dst_offset_ignored": ("        else\n          memcpy(head_vec(dst, p, dst_slots[i], dst_head0 + j),",
                                 "        else\n          memcpy(head_vec(dst, p, dst_slots[i], j),"),
    "heads_buffer_row_of_whole_pool": ("uint8_t *b = buf + (((int64_t)p * n + i) * n_heads + j) * hb;",
                                       "uint8_t *b = buf + (((int64_t)p * n + i) * shape->kv_heads + j) * hb;"),
    "mla_latent_plane_ignored": ("return pool->kv_planes == 1 ? 1 : 2;", "return 2;"),
    "mla_counted_as_k_and_v": ("return (int64_t)num_layers * (latent_dim + rope_dim) * elem_bytes;",
                               "return (int64_t)2 * num_layers * (latent_dim + rope_dim) * elem_bytes;"),
    "owner_check_on_source_page": ("if (page_epochs[dst_slots[i] / epoch_page] != epoch) continue;",
                                   "if (page_epochs[src_slots[i] / epoch_page] != epoch) continue;"),
    "owner_check_dropped": ("if (page_epochs[dst_slots[i] / epoch_page] != epoch) continue;", ""),
    "reshard_adjacent_parts_refused": ("q->dst_head0 < parts[m].dst_head0 + parts[m].n_heads)",
                                       "q->dst_head0 <= parts[m].dst_head0 + parts[m].n_heads)"),
    "reshard_one_writer_check_dropped": ("for (int32_t m = 0; m < k; ++m) /* one writer",
                                         "for (int32_t m = 0; m < 0; ++m) /* one writer"),
    "reshard_first_dst_pool_checked_only": ("for (int32_t k = 0; k < n_dsts; ++k)\n    if ((rc = kvxo_check_slots(dsts[k]",
                                            "for (int32_t k = 0; k < 1; ++k)\n    if ((rc = kvxo_check_slots(dsts[k]"),
    "reshard_head_offsets_swapped": ("src_slots, q->src_head0, dsts[q->dst], dst_slots,\n                         q->dst_head0,",
                                     "src_slots, q->dst_head0, dsts[q->dst], dst_slots,\n                         q->src_head0,"),
    "transfer_src_dst_swapped": ("memcpy(head_vec(dst, p, dst_slots[i], h), head_vec(src, p, src_slots[i], h),",
                                 "memcpy(head_vec(src, p, src_slots[i], h), head_vec(dst, p, dst_slots[i], h),"),
}


def _build_mutant(name, old, new, tmp):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for {name} not unique/missing"
    d = os.path.join(tmp, name)
    os.makedirs(d)
    shutil.copy(HDR, d)
    src = os.path.join(d, "kvx_oracle.c")
    open(src, "w").write(text.replace(old, new))
    return oracle.build(src=src, out=os.path.join(d, "libmut.so"))


_CHILD = r"""
import json, sys
sys.path.insert(0, sys.argv[2])
import oracle
from tests import pins
lib = oracle.load(sys.argv[1])
failed = []
for pin in pins.ALL_PINS:
    try:
        pin(lib)
    except AssertionError:
        failed.append(pin.__name__)
print(json.dumps(failed))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    """A mutant may write out of bounds (that is the mistake), so its pins run in a child
    process; the child dying of the corruption also counts as caught."""
    old, new = MUTANTS[name]
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with tempfile.TemporaryDirectory() as tmp:
        path = _build_mutant(name, old, new, tmp)
        res = subprocess.run([sys.executable, "-c", _CHILD, path, root], capture_output=True,
                             text=True, timeout=600)
        if res.returncode != 0:
            return  # crashed on its own planted mistake
        failed = json.loads(res.stdout.strip().splitlines()[-1])
        assert failed, f"planted mistake {name} passed every pin"
