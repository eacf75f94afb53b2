"""bench.py's host logic on the CPU: the ncu traffic lines it reads from the
committed profile summaries (kept only for the current kernel sources), the
roofline entry that carries them, and the backward kernel names it reports."""
import types


def test_profiled_traffic_keeps_lines_of_current_sources(tmp_path, monkeypatch):
    import bench
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "a.md").write_text(
        "# summary\n\n"
        "`traffic: lse_merge_kernel wl merge 123 cur`\n"          # kept
        "`traffic: lse_merge_kernel wl permute 456 old`\n"        # other sources: dropped
        "`traffic: not_a_kernel wl merge 7 cur`\n"                # unknown kernel: dropped
        "`traffic: lse_merge_kernel wl 9 cur`\n"                  # malformed: dropped
        "traffic: attn_fwd_tc_kernel wl2 fwd 1e9 cur\n")          # without backticks: kept
    (prof / "b.txt").write_text("traffic: lse_merge_kernel wl merge 1 cur\n")   # not a summary
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_sha", lambda kernel: "cur")
    assert bench.profiled_traffic() == {("lse_merge_kernel", "wl", "merge"): 123.0,
                                        ("attn_fwd_tc_kernel", "wl2", "fwd"): 1e9}


def test_source_sha_tracks_the_kernel_file():
    import bench
    a = bench.source_sha("attn_fwd_tc_kernel")
    assert len(a) == 12 and a == bench.source_sha("attn_fwd_tc_kernel")
    assert a != bench.source_sha("lse_merge_kernel")
    # the backward's kernels share one source file
    assert (bench.source_sha("attn_bwd_dkdv_tc_kernel")
            == bench.source_sha("attn_bwd_dkdv_tc_kernel+attn_bwd_dq_cached_kernel"))


def test_roof_entry_takes_traffic_of_its_kernel_workload_and_leg():
    import bench
    wl = bench.CONFIGS[2].name
    tm = {("lse_merge_kernel", wl, "merge"): 5.0e8}
    e = bench.roof_entry("lse_merge_kernel", 2, "merge", "hbm", 6000.0, 6778.0, "GB/s", 1.2e9,
                         "bytes", 1, tm)
    assert e["traffic"] == 5.0e8 and abs(e["frac"] - 6000.0 / 6778.0) < 1e-12
    assert e["algorithmic_per_launch"] == 1.2e9
    e = bench.roof_entry("lse_merge_kernel", 2, "permute", "hbm", 1.0, 2.0, "GB/s", 1.0,
                         "bytes", 2, tm)
    assert e["traffic"] is None and e["traffic_unit"] is None and e["algorithmic_per_launch"] == 0.5


def test_backward_kernel_names_follow_the_ds_cache():
    import bench
    assert bench.bwd_kernels(types.SimpleNamespace(ds_cache_bytes=0)) == \
        "attn_bwd_dkdv_tc_kernel+attn_bwd_dq_tc_kernel"
    assert bench.bwd_kernels(types.SimpleNamespace(ds_cache_bytes=1 << 30)) == \
        "attn_bwd_dkdv_tc_kernel+attn_bwd_dq_cached_kernel"
    assert bench.ds_cache_record(types.SimpleNamespace(dq=None)) is None
