"""The DRAM traffic bench.py reports comes from committed ncu records, each keyed by a hash
of the code of the sources its pass compiles. The hash must ignore comments and layout (a
reworded comment does not change what the kernel reads from DRAM) and must follow any
change to the code itself."""

import json
import os

import bench


def test_code_only_drops_comments_and_layout():
    src = 'int a = 1; // note\n/* block\n comment */ float  b =\n 2.0f;\n'
    assert bench._code_only(src) == "int a = 1; float b = 2.0f;"


def test_code_only_keeps_literals():
    src = 'const char* s = "x // y /* z */";\nchar c = \'/\'; char e = \'\\\'\';\n'
    assert bench._code_only(src) == 'const char* s = "x // y /* z */"; char c = \'/\'; char e = \'\\\'\';'


def test_code_only_sees_code_edits():
    a = bench._code_only("x = y + 1; // add one")
    b = bench._code_only("x = y + 2; // add one")
    assert a != b


def test_records_name_existing_sources_and_parse():
    for which, fname in bench.TRAFFIC_RECORDS.items():
        assert which in bench.KERNEL_SOURCES
        for src in bench.KERNEL_SOURCES[which]:
            assert os.path.isfile(os.path.join(bench.ROOT, "exact_attention_23_gb300", "csrc",
                                               src)), src
        with open(os.path.join(bench.ROOT, "profiles", fname)) as f:
            rec = json.load(f)
        assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
        assert len(rec["kernel_source_sha256"]) == 64
