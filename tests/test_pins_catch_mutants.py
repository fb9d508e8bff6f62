"""Planted mistakes in the oracle: each one must fail a pin.

Each mutant is a copy of ``oracle/`` with one plausible mistake written into
it (a wrong head map, an offset off by one, a flipped exponent sign, a partial
block cached, ...).  The oracle's pin tests (``tests/test_oracle_*.py``: the
pages' worked examples, closed forms, invariants and brute force) run against
the copy in a child process.  The unchanged copy must pass them all and every
mutant must fail at least one; a mutant that passes names a pin that is
missing.  Everything runs on the CPU; nothing here touches the CUDA library.

Where a snippet occurs more than once in a file, the first occurrence is
changed (in ``pa_oracle.c`` that is the plain decode).
"""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = sorted(p for p in glob.glob(os.path.join(ROOT, "tests", "test_oracle_*.py"))
              if os.path.abspath(p) != os.path.abspath(__file__))
# set in the child processes: a child never starts mutants of its own
_CHILD = "PA_PINS_MUTANT_CHILD"

C, BM, PC, BK = "pa_oracle.c", "block_manager.py", "prefix_cache.py", "bookkeeping.py"

# (file in oracle/, text, replacement, what the mistake is)
MUTANTS = [
    # address translation and slots
    (C, "*off = pos % B;", "*off = (pos + 1) % B;", "translate: offset one slot late"),
    (C, "*slot = (int64_t)phys * B + off;", "*slot = (int64_t)off * B + phys;", "slot: block and offset transposed"),
    (C, "if (positions[t] < 0) { out[t] = -1; continue; }", "if (positions[t] < 0) { out[t] = 0; continue; }",
     "slot mapping: padding mapped to slot 0"),
    # decode
    (C, "const int kvh = h / G;", "const int kvh = h % Hkv;", "decode: query head h reads KV head h mod Hkv"),
    (C, "z[i] = exp(z[i] - m);", "z[i] = exp(m - z[i]);", "decode: exponent sign flipped"),
    (C, "z[i] = scale * dot;", "z[i] = dot;", "decode: scale dropped"),
    (C, "Vc[(size_t)i * D + d] = load_elem(v_cache, base + d, dtype);",
     "Vc[(size_t)i * D + d] = load_elem(k_cache, base + d, dtype);", "gather: values read from the key cache"),
    (C, "for (int i = 0; i < len; ++i)\n                for (int d = 0; d < D; ++d)\n                    o[d] += z[i]",
     "for (int i = 0; i < len - 1; ++i)\n                for (int d = 0; d < D; ++d)\n                    o[d] += z[i]",
     "decode: last value dropped"),
    # widening of the storage types
    (C, "ldexp((double)(f | 0x400), e - 25)", "ldexp((double)(f | 0x400), e - 24)", "f16: exponent bias off by one"),
    (C, "ldexp((double)f, -24)", "ldexp((double)f, -23)", "f16: subnormal scale wrong"),
    (C, "(uint32_t)b << 16", "(uint32_t)b << 15", "bf16: wrong shift"),
    # partitioned form and its merge
    (C, "const int i1 = (i0 + partition_size < len) ? i0 + partition_size : len;",
     "const int i1 = (i0 + partition_size < len) ? i0 + partition_size - 1 : len;",
     "partitions: last token of each full partition dropped"),
    (C, "den += c * lb[b];", "den += lb[b];", "merge: partition sums not rescaled"),
    (C, "o[d] += c * accb[(size_t)b * D + d];", "o[d] += accb[(size_t)b * D + d];",
     "merge: partition accumulators not rescaled"),
    # chunk attention
    (C, "const size_t tok = (size_t)query_start[s] + t;", "const size_t tok = (size_t)query_start[s] + (n - 1 - t);",
     "chunk: query rows reversed"),
    (C, "for (int h = kvh * G; h < (kvh + 1) * G; ++h)", "for (int h = kvh; h < Hq; h += Hkv)",
     "chunk: strided head grouping"),
    (C, "const int pos = len - n + t;", "const int pos = len - 1;", "chunk: every query sees the whole context"),
    # cache operations
    (C, "const int64_t off = slot % B;", "const int64_t off = (slot + 1) % B;", "write_kv: offset one slot late"),
    (C, "        memmove((char *)v_cache + (size_t)dst * blk, (const char *)v_cache + (size_t)src * blk, blk);\n",
     "", "copy_blocks: values not copied"),
    (C, "memcpy((char *)to_v + (size_t)dst * blk, (const char *)from_v + (size_t)src * blk, blk);",
     "memcpy((char *)to_v + (size_t)dst * blk, (const char *)from_k + (size_t)src * blk, blk);",
     "swap_blocks: values taken from the keys"),
    # block manager
    (BM, "self.ref[s.table[-1]] > 1", "self.ref[s.table[-1]] >= 1", "allocator: copy-on-write of unshared blocks"),
    (BM, "self.ref[old] -= 1 ", "self.ref[old] -= 0 ", "allocator: copy-on-write keeps the shared reference"),
    (BM, "for b in p.table:\n            self.ref[b] += 1", "for b in p.table:\n            self.ref[b] += 0",
     "allocator: fork takes no references"),
    (BM, "grow = -(-(s.length + n) // B) - (-(-s.length // B))", "grow = (s.length + n) // B - s.length // B",
     "allocator: growth counted with floor"),
    (BM, "if self.ref[b] == 0:", "if self.ref[b] <= 1:", "allocator: block freed while still held"),
    (BM, "self.free.append(b)", "self.free.appendleft(b)", "allocator: freed blocks reused first"),
    (BM, "        host.seqs[hid].length = s.length\n        self.free_seq(sid)\n",
     "        host.seqs[hid].length = s.length\n", "swap out: device blocks kept"),
    # prefix cache
    (PC, "victim = min(leaves", "victim = max(leaves", "prefix cache: most recently used evicted"),
    (PC, "self.bm.ref[self.entries[p][0]] == 1]", "self.bm.ref[self.entries[p][0]] >= 1]",
     "prefix cache: blocks in use evicted"),
    (PC, "m = min(len(blocks), len(tokens) // self.B)", "m = min(len(blocks), -(-len(tokens) // self.B))",
     "prefix cache: partial blocks cached"),
    (PC, "            e[1] = self.clock\n", "", "prefix cache: a lookup does not count as a use"),
    # bookkeeping arithmetic
    (BK, "return (tokens + block_size - 1) // block_size", "return tokens // block_size + 1",
     "bookkeeping: blocks counted as floor + 1"),
    (BK, "return 2 * layers * heads * head_dim * dtype_bytes", "return layers * heads * head_dim * dtype_bytes",
     "bookkeeping: keys only"),
    (BK, "return 1 - Fraction(block_size - 1) / Fraction(mean_len)",
     "return 1 - Fraction(block_size) / Fraction(mean_len)", "bookkeeping: utilisation bound off by one"),
    (BK, "shared = prompt // block_size\n", "shared = blocks_for(prompt, block_size)\n",
     "bookkeeping: partial prompt block shared"),
    (BK, '"paged_frag": Fraction(paged - tokens, paged)', '"paged_frag": Fraction(paged - tokens, tokens)',
     "bookkeeping: fragmentation over tokens"),
    (BK, "private = blocks_for(suffix, block_size)", "private = blocks_for(prompt % block_size + suffix, block_size)",
     "bookkeeping: shared partial block also stored per request"),
    (BK, '"reduction": Fraction(naive, paged)', '"reduction": Fraction(paged, naive)', "bookkeeping: reduction inverted"),
    (BK, "naive = max_len * len(lengths)", "naive = max_len * len(lengths) + 1", "bookkeeping: reserved slots off by one"),
    (BK, "without = per_req_unshared * requests", "without = per_req_unshared * requests - 1",
     "bookkeeping: unshared total off by one"),
    (BK, "return Fraction(tokens, slots) if slots else Fraction(1)",
     "return Fraction(tokens, slots + 1) if slots else Fraction(1)", "bookkeeping: utilisation over one slot too many"),
    (BK, "return prompt // block_size", "return -(-prompt // block_size)", "bookkeeping: partial block counted as shareable"),
    # refusals and the less travelled paths (each mutant stays inside its buffers
    # on the inputs the pins give it)
    (C, "if (Hq % Hkv != 0 || dtype < 0 || dtype > 2)", "if (dtype < 0 || dtype > 2)",
     "oracle: query heads not a multiple of KV heads accepted"),
    (C, "if (positions[t] / B >= max_blocks)\n            return -1;", "if (positions[t] / B > max_blocks)\n            return -1;",
     "slot mapping: position past the table accepted"),
    (C, "if (B <= 0 || pos < 0)\n        return -1;", "if (B <= 0)\n        return -1;", "slot: negative position accepted"),
    (C, "if (n < 0 || n > lens[s])", "if (n < 0)", "chunk: more queries than context accepted"),
    (BM, "self.seqs[sid].length = p.length", "self.seqs[sid].length = 0", "allocator: fork starts empty"),
    (BM, "if n < 0:\n            raise ValueError", "if n < -1:\n            raise ValueError", "allocator: negative append accepted"),
    (BM, "cow = n > 0 and s.length % B != 0", "cow = s.length % B != 0", "allocator: empty append copies on write"),
    (BM, "shared = sum(1 for r in self.ref if r > 1)", "shared = sum(1 for r in self.ref if r >= 1)",
     "allocator: used blocks counted as shared"),
    (BM, "\"padded_slots\": slots - tokens}", "\"padded_slots\": slots}", "allocator: padding counted as all slots"),
    (BM, "        self.seqs[sid].length = hs.length\n        host.free_seq(hid)\n", "        self.seqs[sid].length = hs.length\n",
     "swap in: host blocks kept"),
    (BM, "if len(s.table) > len(host.free)", "if len(s.table) > len(host.free) + 1", "swap out: host pool overdrawn"),
    (BM, "        if self._fail_budget is not None:\n            self._fail_budget -= 1\n", "",
     "allocator: injected failure never comes"),
    (PC, "if len(set(new)) != len(new) or any(b in held for b in new):", "if any(b in held for b in new):",
     "prefix cache: one block cached under two prefixes"),
    (PC, "or self.bm.ref[int(b)] < 1 for b in blocks[:m]", "for b in blocks[:m]", "prefix cache: free block cached"),
    (PC, "self.bm.ref[int(blocks[k - 1])] += 1\n                added += 1", "added += 1",
     "prefix cache: cache takes no reference"),
    (PC, "bm.seqs[sid].length = len(blocks) * bm.B", "bm.seqs[sid].length = len(blocks) * bm.B - 1",
     "prefix cache: sequence from a prefix one token short"),
    (PC, "    for b in blocks:\n        bm.ref[int(b)] += 1\n", "", "prefix cache: sequence from a prefix takes no references"),
    # extreme logits, widening edge cases, and more refusals
    (C, "double m = -INFINITY;\n                for (int i = i0; i < i1; ++i) {",
     "double m = 0.0;\n                for (int i = i0; i < i1; ++i) {", "partitions: maximum started at 0"),
    (C, "double mstar = mb[0];", "double mstar = mb[nparts - 1];", "merge: m* from the last partition only"),
    (C, "double m = z[0];\n            for (int i = 1; i < len; ++i)", "double m = z[len - 1];\n            for (int i = 1; i < len - 1; ++i)",
     "decode: maximum misses the first and last logits"),
    (C, "mag = f ? NAN : INFINITY;", "mag = INFINITY;", "f16: NaN widened to infinity"),
    (C, "return sign ? -mag : mag;", "return mag;", "f16: sign dropped"),
    (C, "T < 0 || query_start[0] != 0 ||", "T < 0 || query_start[0] < 0 ||", "chunk: ranges not starting at row 0 accepted"),
    (C, "if (n < 0 || n > lens[s])\n            return -1;", "if (n < 0 || n > lens[s] + 1)\n            return -1;",
     "chunk: one query more than the context accepted"),
    (C, "const size_t blk = (size_t)Hkv * B * D * elem_size(dtype);\n    for (int p = 0; p < P; ++p) {\n"
        "        const int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];\n        if (src < 0 || src >= N",
     "const size_t blk = (size_t)Hkv * B * D * elem_size(dtype) / 2;\n    for (int p = 0; p < P; ++p) {\n"
     "        const int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];\n        if (src < 0 || src >= N",
     "copy_blocks: half of each block"),
    (BM, "self.free = deque(order)", "self.free = deque(sorted(order))", "allocator: free order ignored"),
    (BM, "self.cow_copies += 1", "self.cow_copies += 0", "allocator: copies not counted"),
    (BM, "if num_blocks <= 0 or block_size <= 0:", "if num_blocks < 0 or block_size <= 0:", "allocator: empty pool accepted"),
    (BM, "if sorted(order) != list(range(num_blocks)):", "if len(order) != num_blocks:",
     "allocator: free order not checked as a permutation"),
    (PC, "while k * self.B <= len(tokens):", "while k * self.B < len(tokens):",
     "prefix cache: a prompt ending on a block boundary loses its last block"),
    (BK, "if tokens < 0 or block_size <= 0:", "if block_size <= 0:", "bookkeeping: negative token count accepted"),
    (BK, '"naive_frag": Fraction(naive - tokens, naive)', '"naive_frag": Fraction(naive - tokens, paged)',
     "bookkeeping: reserved-slot fragmentation over paged slots"),
]

# Loads the oracle copy given as argv[1] before pytest can put the repository
# first on sys.path, then runs the pin tests given after it.
_DRIVER = r"""
import sys
sys.path.insert(0, sys.argv[1])
import oracle, oracle.block_manager, oracle.prefix_cache, oracle.bookkeeping
for m in (oracle, oracle.block_manager, oracle.prefix_cache, oracle.bookkeeping):
    assert m.__file__.startswith(sys.argv[1]), m.__file__
import pytest
sys.exit(pytest.main(["-q", "-x", "-p", "no:cacheprovider", *sys.argv[2:]]))
"""


def _run_pins(workdir, mutant):
    """Copy oracle/ into workdir, plant `mutant` (None: no change), run the pins."""
    dst = os.path.join(workdir, "oracle")
    shutil.copytree(os.path.join(ROOT, "oracle"), dst, ignore=shutil.ignore_patterns("_build", "__pycache__"))
    if mutant is not None:
        name, old, new, what = mutant
        path = os.path.join(dst, name)
        with open(path) as f:
            src = f.read()
        if old not in src:
            return None, f"stale mutant ({what}): text not found in {name}"
        with open(path, "w") as f:
            f.write(src.replace(old, new, 1))
    r = subprocess.run([sys.executable, "-c", _DRIVER, workdir, *PINS], capture_output=True, text=True,
                       timeout=600, cwd=workdir, env=dict(os.environ, **{_CHILD: "1"}))
    return r.returncode, (r.stdout + r.stderr)[-2000:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    if os.environ.get(_CHILD):
        pytest.skip("inside a mutant run")
    if not shutil.which("gcc"):
        pytest.skip("gcc not found")
    cases = [None] + MUTANTS
    dirs = [str(tmp_path_factory.mktemp(f"mutant{i}")) for i in range(len(cases))]
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(_run_pins, dirs, cases))
    return {None if c is None else c[3]: r for c, r in zip(cases, results)}


def test_unchanged_copy_passes_every_pin(outcomes):
    rc, log = outcomes[None]
    assert rc == 0, log


@pytest.mark.parametrize("what", [m[3] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(outcomes, what):
    rc, log = outcomes[what]
    assert rc is not None, log
    # 1: tests ran and at least one failed (not a crash or a collection error)
    assert rc == 1, f"{what}: exit status {rc}\n{log}"
