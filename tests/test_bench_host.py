"""Host logic of bench.py that decides whether a committed ncu traffic figure
still describes the kernel: the per-workload source hash."""
import bench

DEC = open(bench.os.path.join(bench.ROOT, "paged_gqa_decode_02_gb300", "csrc", "pa_decode_kernels.cuh")).read()
COM = open(bench.os.path.join(bench.ROOT, "paged_gqa_decode_02_gb300", "csrc", "pa_common.cuh")).read()
SEP = "// " + "-" * 66 + " "


def _h(w, dec=DEC, com=COM):
    return bench.kernel_source_hash(w, dec, com)


def test_defaults_read_the_tree():
    for w in bench._USES:
        assert bench.kernel_source_hash(w) == _h(w)


def test_comments_and_blank_lines_do_not_change_the_hash():
    edited = DEC.replace("namespace pa {", "// a new comment line\n\nnamespace pa {  /* and a block\ncomment */", 1)
    assert edited != DEC
    for w in bench._USES:
        assert _h(w, edited) == _h(w)


def test_code_changes_do_change_the_hash():
    edited = DEC.replace("constexpr int kMaxSegs = 64;", "constexpr int kMaxSegs = 65;", 1)
    assert edited != DEC
    for w in bench._USES:
        assert _h(w, edited) != _h(w)
    assert _h("qwen25_7b_bf16", com=COM + "\nint x;\n") != _h("qwen25_7b_bf16")


def test_string_contents_are_not_taken_for_comments():
    assert bench._code_only('asm("a // b");') == 'asm("a // b");'
    assert bench._code_only('asm("a /* b */ c");') == 'asm("a /* b */ c");'
    assert bench._code_only("x = '/'; // c") == "x = '/';"


def test_a_consumer_section_only_reaches_its_own_workloads():
    head = SEP + "consumer math (tensor cores, uint4 KV)\n"
    assert DEC.count(head) == 1
    edited = DEC.replace(head, head + "static int unused_by_bf16 = 1;\n", 1)
    assert _h("qwen25_7b_bf16", edited) == _h("qwen25_7b_bf16")
    assert _h("qwen3_8b_int8", edited) == _h("qwen3_8b_int8")
    assert _h("long_uint4", edited) != _h("long_uint4")
