"""The kernel-source hash that keys bench.py's DRAM-traffic table: blind to comments, not to code."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_comments_are_dropped_and_literals_kept():
    src = 'int a = 1; // note\n/* block\n comment */ const char* s = "x//y /* z */"; char q = \'\\\'\';'
    assert bench.strip_comments(src) == 'int a = 1; const char* s = "x//y /* z */"; char q = \'\\\'\';'


def test_comment_edits_keep_the_hash_code_edits_change_it():
    base = "__global__ void k(int* p) {\n  // first\n  p[0] = 1;  /* one */\n}\n"
    recommented = "__global__ void k(int* p) {\n  // a different note\n  p[0] = 1;\n}\n"
    recoded = "__global__ void k(int* p) {\n  // first\n  p[0] = 2;  /* one */\n}\n"
    assert bench.strip_comments(base) == bench.strip_comments(recommented)
    assert bench.strip_comments(base) != bench.strip_comments(recoded)


def test_inline_asm_strings_survive():
    src = 'asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.b64 [%0];" :: "r"(b));  // c'
    assert "tcgen05.commit.cta_group::1" in bench.strip_comments(src)


def test_traffic_entries_name_a_hash():
    for name, (nbytes, digest) in bench.TRAFFIC.items():
        assert nbytes > 0 and len(digest) == 16, name
