"""CPU: the kernel-source hash that ties ncu summaries to the code ignores
comments and layout but not code (bench.py code_only / kernel_source_hash)."""
import bench


def test_comments_and_layout_do_not_count():
    a = 'int f(int x) {  // doubles x\n    return 2 * x; /* twice */\n}\n'
    b = 'int f(int x) {\n  return 2 * x;\n}  // edited comment\n'
    assert bench.code_only(a) == bench.code_only(b)


def test_code_and_string_literals_count():
    a = 'asm volatile("mov.u32 %0, 1; // not a comment" : "=r"(r));'
    b = 'asm volatile("mov.u32 %0, 2; // not a comment" : "=r"(r));'
    assert bench.code_only(a) != bench.code_only(b)
    assert "// not a comment" in bench.code_only(a)
    assert bench.code_only("int x = 1;") != bench.code_only("int x = 2;")
    assert bench.code_only("a b") != bench.code_only("ab")

