"""bench.py host helpers that need no GPU: the kernel-source hash behind the
recorded DRAM traffic ignores comments and layout but not code."""
import bench


def test_strip_comments_keeps_code_and_literals():
    src = ('int a = 1; // trailing\n/* block\n   comment */ const char* s = "x // not a comment";\n'
           "char q = '\\'';  \n\n  /* one */ int b; /* two */\n")
    out = bench.strip_comments(src)
    assert "trailing" not in out and "block" not in out and "one" not in out and "two" not in out
    assert '"x // not a comment"' in out and "'\\''" in out
    assert "int a = 1;" in out and "int b;" in out
    assert "\n\n" not in out and not any(line != line.rstrip() for line in out.splitlines())


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "k.cu").write_text("// header\n__global__ void k(int* p) { p[0] = 1; }\n")
    a = bench.source_sha(["k.cu"])
    (tmp_path / "k.cu").write_text("/* another header */\n__global__ void k(int* p) { p[0] = 1; }  // note\n\n")
    assert bench.source_sha(["k.cu"]) == a
    (tmp_path / "k.cu").write_text("__global__ void k(int* p) { p[0] = 2; }\n")
    assert bench.source_sha(["k.cu"]) != a


def test_stats_median_min_max_and_launch_count():
    s = bench.stats([(3.0, 16), (1.0, 16), (2.0, 16), (10.0, 16)])
    assert s == {"median": 2.5, "min": 1.0, "max": 10.0, "launches": 64}


def test_o0_record_reads_back(tmp_path, monkeypatch):
    from sparse_attention_indexer_02_gb300 import build as qbuild

    rec = tmp_path / "rec.json"
    monkeypatch.setattr(qbuild, "O0_RECORD", str(rec))
    assert qbuild.o0_units() == []
    rec.write_text('["umma_bf16"]')
    assert qbuild.o0_units() == ["umma_bf16"]


def test_reference_arm_line_and_warmup_floor(capsys):
    """The reference arm (the CPU oracle on a bounded sample) prints one JSON
    line with the contract's keys; a warm-up below 3 steps runs as 3 and the
    line reports 3."""
    import json

    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "1", "--workload", "tiny_mtp"])
    line = [x for x in capsys.readouterr().out.splitlines() if x.startswith("{")][-1]
    d = json.loads(line)
    assert d["impl"] == "reference" and d["warmup"] == 3 and d["steps"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
