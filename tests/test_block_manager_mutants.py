"""Plant plausible mistakes in a copy of the host block manager and check that
its CPU tests (test_block_manager.py) catch every one.

Each mutant is a one-line edit of pa_block_manager.cpp. It is compiled on the
CPU and linked with the library's other objects into a separate shared
library, which a subprocess loads in place of the real one. No GPU is used.

A hash hit must be confirmed by the block's token ids; with a 64-bit chain
hash a wrong hit never happens in a test, so that check is exercised by a
build whose hash keeps 4 bits (collisions everywhere): the randomized run
must still pass on it, and must fail once the token check is removed.
"""
import os
import subprocess
import sys

import pytest

from paged_gqa_decode_02_gb300 import build as pbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "paged_gqa_decode_02_gb300", "csrc", "pa_block_manager.cpp")
LIB_DIR = os.path.join(ROOT, "paged_gqa_decode_02_gb300", "_lib")

NARROW_HASH = "-DPA_BM_HASH_MASK=0xFull"
# mutant -> the build flags and the tests it is run against
SUITE = {"unchecked_hash_hit": ([NARROW_HASH], "randomized")}

MUTANTS = {
    "no_copy_on_write": ("const bool cow = sq.len % bs != 0 && bm->blocks[sq.blocks.back()].ref > 1;",
                         "const bool cow = false;"),
    "unchecked_hash_hit": ("return bl.parent == parent && std::equal(bl.tokens.begin(), bl.tokens.end(), tokens) ? it->second : -1;",
                           "return it->second;"),
    "partial_blocks_cached": ("  const int64_t nfull = n_tokens / bs;\n  // leading full blocks",
                              "  const int64_t nfull = nblk;\n  // leading full blocks"),
    "most_recent_reused_first": ("      idle_cached.push_back(b);\n      blocks[b].lru = std::prev(idle_cached.end());",
                                 "      idle_cached.push_front(b);\n      blocks[b].lru = idle_cached.begin();"),
    "fork_without_refs": ("  for (int32_t b : child.blocks) bm->hold(b);\n", ""),
    "swap_in_keeps_slots": ("    bm->cpu_free.push_back(sq.blocks[(size_t)i]);\n    sq.blocks[(size_t)i] = b;",
                            "    sq.blocks[(size_t)i] = b;"),
    "swap_out_keeps_gpu_blocks": ("  for (auto b = sq.blocks.rbegin(); b != sq.blocks.rend(); ++b) bm->release(*b);\n  sq.blocks = std::move(slots);",
                                  "  sq.blocks = std::move(slots);"),
    "swap_in_wrong_slot_order": ("    cpu_src[i] = sq.blocks[(size_t)i];", "    cpu_src[i] = sq.blocks[(size_t)(n - 1 - i)];"),
}


@pytest.fixture(scope="module")
def objects():
    pbuild.build()
    objs = [os.path.join(LIB_DIR, os.path.splitext(f)[0] + ".o") for f in pbuild.SOURCES
            if f != "pa_block_manager.cpp"]
    assert all(os.path.exists(o) for o in objs)
    return objs


def _build_and_run(text, name, objects, tmp_path, flags=(), select=None):
    """Compile `text` as the block manager, link it into a library of its own
    and run the block-manager tests against it; returns the subprocess."""
    src = tmp_path / f"{name}.cpp"
    src.write_text(text)
    obj, lib = tmp_path / f"{name}.o", tmp_path / f"lib_{name}.so"
    subprocess.run(["g++", "-O1", "-std=c++17", "-fPIC", *flags, "-I", os.path.join(ROOT, "include"), "-c",
                    str(src), "-o", str(obj)], check=True)
    subprocess.run([pbuild.NVCC] + pbuild.ARCH + ["-shared", "-o", str(lib)] + objects + [str(obj), "-lcuda"],
                   check=True)
    args = ["-x", "-q", "-p", "no:cacheprovider", os.path.join(ROOT, "tests", "test_block_manager.py")]
    if select:
        args += ["-k", select]
    code = ("import sys; sys.path.insert(0, %r); import paged_gqa_decode_02_gb300.binding as B; B.LIB_PATH = %r; "
            "import pytest; sys.exit(pytest.main(%r))" % (ROOT, str(lib), args))
    return subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)


def test_manager_stays_correct_when_hashes_collide(objects, tmp_path):
    r = _build_and_run(open(SRC).read(), "narrow_hash", objects, tmp_path, [NARROW_HASH], "randomized")
    assert r.returncode == 0, r.stdout[-3000:]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_block_manager_tests_catch_planted_mistake(name, objects, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    flags, select = SUITE.get(name, ((), None))
    r = _build_and_run(text.replace(old, new), name, objects, tmp_path, flags, select)
    assert r.returncode != 0, f"mutant {name} survived the block-manager tests:\n{r.stdout[-2000:]}"
