"""The oracle's pins must catch plausible mistakes: each case below plants one mistake in a copy of
the oracle's C source (on the CPU, in a temporary directory), builds it, runs every pin of
test_oracle_pins.py against it in a child process, and expects at least one pin to fail (or the
child to die). The real oracle is never modified."""
import os
import subprocess
import sys
import tempfile

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

MUTANTS = [
    # (name, text in the oracle, planted replacement)
    ("fnv1_order", "h ^= (uint64_t)data[i];\n        h *= ORACLE_FNV64_PRIME;",
     "h *= ORACLE_FNV64_PRIME;\n        h ^= (uint64_t)data[i];"),
    ("fnv_prime", "1099511628211ULL", "1099511628213ULL"),
    ("parent_big_endian", "(uint8_t)(parent >> (8 * b))", "(uint8_t)(parent >> (8 * (7 - b)))"),
    ("token_big_endian", "(uint8_t)(tok >> (8 * b))", "(uint8_t)(tok >> (8 * (3 - b)))"),
    ("no_chaining", "parent = out[j];", "parent = 0;"),
    ("src_slot_from_dst_bs", "int64_t src_slot = t % src->block_size;", "int64_t src_slot = t % dst->block_size;"),
    ("dst_shard_mapping", "int32_t ds = g / dst->heads_per_shard;", "int32_t ds = g % dst->n_shards;"),
    ("whole_last_block", "for (int64_t t = 0; t < n_tokens[r]; ++t) {",
     "for (int64_t t = 0; t < (n_tokens[r] + dst->block_size - 1) / dst->block_size * dst->block_size; ++t) {"),
    ("runs_cut_on_src_only", "|| (src_ids[i] != src_ids[i - 1] + 1) || (dst_ids[i] != dst_ids[i - 1] + 1);",
     "|| (src_ids[i] != src_ids[i - 1] + 1);"),
    ("token_runs_cut_on_src_only", "if (t == 0 || srow != prev_s + 1 || drow != prev_d + 1) {",
     "if (t == 0 || srow != prev_s + 1) {"),
    ("local_hit_not_prefix", "while (l_loc < n_full && oracle_is_resident(sorted, n_local, h[l_loc])) ++l_loc;",
     "for (int64_t q = 0; q < n_full; ++q) l_loc += oracle_is_resident(sorted, n_local, h[q]);"),
    ("threshold_strict", "(missing > 0 && missing >= threshold)", "(missing > 0 && missing > threshold)"),
    ("missing_not_clipped", "l_rem > l_loc ? l_rem - l_loc : 0", "l_rem - l_loc"),
    ("free_list_offset", "pair_dst[k] = free_blocks[out_dst_start[s] + i];\n            ++k;\n        }",
     "pair_dst[k] = free_blocks[i];\n            ++k;\n        }"),
    ("free_list_offset_holes", "pair_dst[k] = free_blocks[out_dst_start[s] + i];\n                ++k;",
     "pair_dst[k] = free_blocks[i];\n                ++k;"),
    ("remote_span_start", "remote_blk[rem_off[s] + out_local_hit[s] + i]", "remote_blk[rem_off[s] + i]"),
    ("holes_counted_from_prefix", "for (int64_t j = 0; j < l_rem; ++j)\n                if (!oracle_is_resident(sorted, n_local, h[j])) ++missing_blocks;",
     "for (int64_t j = l_loc; j < l_rem; ++j)\n                ++missing_blocks;"),
    ("ttl_strict", "if (expiry && now >= expiry[s]) n_rem = 0;", "if (expiry && now > expiry[s]) n_rem = 0;"),
    ("keep_last_always", "&& l_rem > 0 && l_rem * block_size >= n_tok) --l_rem;", "&& l_rem > 0) --l_rem;"),
    ("hnd_as_nhd", "if (p->layout == 1) return (blk * p->heads_per_shard + head) * p->block_size + slot;",
     "if (p->layout == 1) return (blk * p->block_size + slot) * p->heads_per_shard + head;"),
    ("hnd_slot_head_swapped", "if (p->layout == 1) return (blk * p->heads_per_shard + head) * p->block_size + slot;",
     "if (p->layout == 1) return (blk * p->heads_per_shard + slot) * p->block_size + head;"),
    ("dst_block_from_src_bs", "int64_t dblk = dst_ids[r][t / dst->block_size];",
     "int64_t dblk = dst_ids[r][t / src->block_size];"),
    ("dst_head_is_src_head", "int32_t dh = g % dst->heads_per_shard;", "int32_t dh = h;"),
    ("global_head_from_dst_split", "int32_t g = s * src->heads_per_shard + h;", "int32_t g = s * dst->heads_per_shard + h;"),
    ("src_plane_dropped", "src->base[((int64_t)l * src->n_planes + p) * src->n_shards + s]",
     "src->base[((int64_t)l * src->n_planes) * src->n_shards + s]"),
    ("remote_span_counts_all_matches",
     "while (l_rem < n_full && l_rem < n_rem && h[l_rem] == remote_hash[rem_off[s] + l_rem]) ++l_rem;",
     "for (int64_t q = 0; q < n_full && q < n_rem; ++q) l_rem += h[q] == remote_hash[rem_off[s] + q];"),
    ("remote_span_ignores_published_count", "while (l_rem < n_full && l_rem < n_rem && h[l_rem]",
     "while (l_rem < n_full && h[l_rem]"),
    ("dst_start_session_index", "cursor += out_missing[s] / block_size;", "cursor += 1;"),
]

CHILD = r"""
import sys, inspect
sys.path[:0] = [{root!r}, {here!r}]
import oracle, test_oracle_pins as pins
orc = oracle.Oracle({lib!r})
failed = []
for name, fn in inspect.getmembers(pins, inspect.isfunction):
    if not name.startswith("test_"):
        continue
    marks = getattr(fn, "pytestmark", [])
    params = [m for m in marks if m.name == "parametrize"]
    calls = [dict()]
    for m in params:
        names = [n.strip() for n in m.args[0].split(",")] if isinstance(m.args[0], str) else list(m.args[0])
        new = []
        for c in calls:
            for v in m.args[1]:
                v = v if isinstance(v, (tuple, list)) and len(names) > 1 else (v,)
                new.append(dict(c, **dict(zip(names, v))))
        calls = new
    for kw in calls:
        args = {{k: v for k, v in kw.items()}}
        if "orc" in inspect.signature(fn).parameters:
            args["orc"] = orc
        try:
            fn(**args)
        except Exception as e:
            failed.append(name)
print("FAILED_PINS", sorted(set(failed)))
sys.exit(0 if failed else 1)
"""


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new):
    with open(os.path.join(ROOT, "oracle", "kvx_oracle.c")) as f:
        text = f.read()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, "mutant.c")
        with open(src, "w") as f:
            f.write(text.replace(old, new))
        lib = oracle.build(src=src, out=os.path.join(tmp, "libmutant.so"), extra_flags=["-w"])
        proc = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, here=HERE, lib=lib)],
                              capture_output=True, text=True, timeout=300)
    assert proc.returncode != 1, f"no pin caught the planted mistake {name}: {proc.stdout[-2000:]}"


def test_unmodified_oracle_passes_every_pin_in_child():
    """Control: the harness above must report no failed pin for the real oracle source."""
    with tempfile.TemporaryDirectory() as tmp:
        lib = oracle.build(out=os.path.join(tmp, "libcontrol.so"), extra_flags=["-w"])
        proc = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, here=HERE, lib=lib)],
                              capture_output=True, text=True, timeout=300)
    assert proc.returncode == 1 and "FAILED_PINS []" in proc.stdout, proc.stdout[-2000:] + proc.stderr[-2000:]
