"""CPU checks of bench.py's bookkeeping: the code hash that decides whether a
committed ncu summary still describes the kernel it was taken on."""
from __future__ import annotations

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_comments_do_not_change_the_code_hash():
    a = 'int f(int x) {\n  return x + 1;  // one\n}\n'
    b = '// header\n/* block\n   comment */\nint f(int x) {\n\n  return x + 1;\n}\n'
    assert bench._code_only(a) == bench._code_only(b)


def test_code_changes_do_change_the_code_hash():
    a = 'int f(int x) { return x + 1; }\n'
    b = 'int f(int x) { return x + 2; }\n'
    assert bench._code_only(a) != bench._code_only(b)


def test_strings_keep_their_contents():
    src = 'asm("ld.shared.v4.u32 {%0}, [%1];"); // tail\n'
    assert bench._code_only(src) == 'asm("ld.shared.v4.u32 {%0}, [%1];");'
