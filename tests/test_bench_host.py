"""Host logic of bench.py, checked on the CPU: the code-only source hash that
ties a committed ncu capture (profiles/ncu_traffic.json) to the kernel sources
it was taken on."""
from __future__ import annotations

import bench


SRC = '''// header comment
#include "x.h"  // trailing comment
/* block
   comment */
__global__ void k(float *p) {
    asm volatile("ld.global.f32 %0, [%1]; // not a comment" : "=f"(p[0]) : "l"(p));

    p[1] = 2.f;  /* inline */ p[2] = 3.f;
}
'''


def test_code_only_drops_comments_and_blank_lines():
    code = bench._code_only(SRC)
    assert "header comment" not in code and "trailing comment" not in code
    assert "block" not in code and "inline" not in code
    assert '"ld.global.f32 %0, [%1]; // not a comment"' in code  # string literals kept whole
    assert "p[1] = 2.f;" in code and "p[2] = 3.f;" in code
    assert "\n\n" not in code


def test_comment_edits_keep_the_code_and_code_edits_change_it():
    edited_comment = SRC.replace("// header comment", "// another header").replace("/* inline */", "")
    assert bench._code_only(edited_comment) == bench._code_only(SRC)
    edited_code = SRC.replace("p[1] = 2.f;", "p[1] = 4.f;")
    assert bench._code_only(edited_code) != bench._code_only(SRC)


def test_kernel_source_hash_is_stable():
    assert bench.kernel_source_hash() == bench.kernel_source_hash()
    assert len(bench.kernel_source_hash()) == 16
