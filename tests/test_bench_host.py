"""Host-side pieces of bench.py that decide what a bench line reports: the
source digest that keeps a recorded ncu traffic figure tied to the kernel it
was taken on (comments do not count, code does), and the record lookup."""
import bench


KERNEL = '''
// a kernel
__global__ void k(int *x) {
  /* block
     comment */
  x[threadIdx.x] = 1;  // trailing
}
'''


def test_comments_and_layout_do_not_change_the_code():
    reworded = KERNEL.replace("// a kernel", "// the same kernel, described differently")
    reworded = reworded.replace("/* block\n     comment */", "/* another\n comment */")
    relaid = "\n\n".join(line.strip() for line in KERNEL.splitlines())
    assert bench.code_only(reworded) == bench.code_only(KERNEL)
    assert bench.code_only(relaid) == bench.code_only(KERNEL)


def test_code_edits_change_the_code():
    assert bench.code_only(KERNEL.replace("= 1;", "= 2;")) != bench.code_only(KERNEL)
    assert bench.code_only(KERNEL.replace("int *x", "int *y")) != bench.code_only(KERNEL)
    assert "comment" not in bench.code_only(KERNEL) and "trailing" not in bench.code_only(KERNEL)


def test_traffic_record_lookup(tmp_path, monkeypatch):
    # a record is reported for its kernel and workload while that kernel's
    # sources hash to its digest, and for nothing else
    kern = "pkv_decode_tc_kernel<128, bf16, append>"
    wide = "pkv_decode_wide_kernel<256, bf16>"
    (tmp_path / "profiles").mkdir()
    rec = tmp_path / "profiles" / "decode_traffic.txt"
    digests = {k: bench.sources_sha256(k) for k in (kern, wide)}   # of the sources in this tree
    assert digests[kern] != digests[wide]

    def write(sha_tc, sha_wide):
        rec.write_text("# captures\n%s | llama8b_bf16 | %s | 714866688\n"
                       "%s | mqa_bf16 | %s | 161000000\n" % (kern, sha_tc, wide, sha_wide))

    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "sources_sha256", lambda k="": digests[k])
    write(digests[kern], digests[wide])
    assert bench.decode_traffic(kern, "llama8b_bf16") == 714866688
    assert bench.decode_traffic(wide, "mqa_bf16") == 161000000
    assert bench.decode_traffic(kern, "long_bf16") is None
    assert bench.decode_traffic(wide, "llama8b_bf16") is None
    write("0" * 64, digests[wide])           # the tensor-core kernel changed since
    assert bench.decode_traffic(kern, "llama8b_bf16") is None
    assert bench.decode_traffic(wide, "mqa_bf16") == 161000000


def test_kernel_sources_cover_every_decode_kernel():
    import os
    for fam, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(bench.ROOT, "paged_kv_cache_67_gb300", "csrc", f))
        assert len(bench.sources_sha256(fam + "<x>")) == 64
