"""Host-side pieces of bench.py that decide what the JSON line reports: the
code-text hash that keeps an ncu traffic record valid only for the kernel
code it was measured on, and the algorithmic byte count of a decode step."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_text_drops_comments_and_layout_only():
    a = "int f(int x) {\n    // twice\n    return 2 * x; /* doubled */\n}\n"
    b = "int f(int x){return 2*x;}"
    assert bench.code_text(a) == bench.code_text(b)
    # a code edit changes it
    assert bench.code_text(a) != bench.code_text(a.replace("2 * x", "3 * x"))
    # comment markers inside string literals are code, escapes included
    s = 'const char *p = "// not a comment \\" /* nor this */";'
    assert bench.code_text(s) == 'constchar*p="// not a comment \\" /* nor this */";'


def test_traffic_records_match_the_kernels_in_tree():
    """Every recorded capture names a kernel file that exists; a record whose
    code hash no longer matches reports no traffic rather than a stale one."""
    for (kfile, workload), rec in bench.NCU_TRAFFIC.items():
        h = bench.source_hash(kfile)
        got = bench.traffic_for(kfile, workload)
        assert got == (rec["bytes"] if h == rec["src"] else None)


def test_decode_algorithmic_bytes_count_shared_blocks_once():
    from workloads import decode_config
    c = decode_config(1)
    total = bench.decode_alg_bytes(c)
    kv = c.unique_kv_bytes()
    assert total > kv  # q, out, new rows and the table come on top
    assert total < 2 * kv + 10 * c.q.numel() * c.q.element_size()
