"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every
symbol the header declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from kv_cache_tempcache_gb300 import build_lib, _lib
    build_lib.build()
    return _lib.load()


def header_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(fastar_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    from kv_cache_tempcache_gb300 import _lib
    names = header_symbols()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.symbols(), f"{n} has no Python binding"


def test_status_strings_and_version(lib):
    from kv_cache_tempcache_gb300 import _lib
    assert _lib.version() >= 100
    for code in (0, -1, -2, -3, -4, -5):
        assert _lib.status_string(code) != "unknown status"
    assert _lib.status_string(-99) == "unknown status"


def test_workspace_sizes(lib):
    from kv_cache_tempcache_gb300 import _lib
    assert _lib.workspace_bytes(_lib.OP_MATCH, 12, 4680, 9360) >= 12 * 4680 * 16
    assert _lib.workspace_bytes(_lib.OP_SPARSE_ATTN, 12, 4680, 9360, 128, 64, 2) >= 12 * 4680 * 2 * 129 * 4
    assert _lib.workspace_bytes(_lib.OP_ANNCA, 12, 0, 0, 128, 64, 2, 512, 3) >= 12 * 3 * 512 * 4
    assert _lib.workspace_bytes(99, 12, 10) == 0


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below fails validation first


def test_argument_validation_rejects_before_launch(lib):
    from kv_cache_tempcache_gb300 import _lib as L
    s = None
    # unsupported dtype / head dim
    assert lib.fastar_bucket_assign(FAKE, 7, 1, 8, 128, 1024, 128, FAKE, 4, 1, FAKE, None, None, s) == L.EUNSUPPORTED
    assert lib.fastar_bucket_assign(FAKE, L.BF16, 1, 8, 96, 1024, 96, FAKE, 4, 1, FAKE, None, None, s) == L.EUNSUPPORTED
    # r > B, B too large
    assert lib.fastar_bucket_assign(FAKE, L.BF16, 1, 8, 128, 1024, 128, FAKE, 4, 5, FAKE, None, None, s) == L.ECAPACITY
    assert lib.fastar_bucket_assign(FAKE, L.BF16, 1, 8, 128, 1024, 128, FAKE, 300, 1, FAKE, None, None, s) == L.ECAPACITY
    # misaligned base / stride
    assert lib.fastar_bucket_assign(FAKE + 2, L.BF16, 1, 8, 128, 1024, 128, FAKE, 4, 1, FAKE, None, None, s) == L.EINVAL
    assert lib.fastar_bucket_assign(FAKE, L.BF16, 1, 8, 128, 1024, 129, FAKE, 4, 1, FAKE, None, None, s) == L.EINVAL
    # null output
    assert lib.fastar_bucket_assign(FAKE, L.BF16, 1, 8, 128, 1024, 128, FAKE, 4, 1, None, None, None, s) == L.EINVAL
    # M < Nq
    assert lib.fastar_cache_compact(L.BF16, 1, 100, 128, 50, FAKE, FAKE, 12800, 128, FAKE, FAKE, FAKE, FAKE, FAKE,
                                    FAKE, FAKE, FAKE, FAKE + 16, FAKE + 16, FAKE + 16, FAKE + 16, FAKE, FAKE, None,
                                    s) == L.ECAPACITY
    # in-place compaction is refused
    assert lib.fastar_cache_compact(L.BF16, 1, 10, 128, 50, FAKE, FAKE, 1280, 128, FAKE, FAKE, FAKE, FAKE, FAKE,
                                    FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, s) == L.EINVAL
    # workspace too small
    assert lib.fastar_tempcache_match(FAKE, FAKE, L.BF16, 1, 64, 128, 8192, 128, FAKE, FAKE, FAKE, 128, 0.9, FAKE,
                                      None, None, FAKE, None, None, FAKE, 16, s) == L.EWORKSPACE
    assert lib.fastar_sparse_attn(FAKE, L.BF16, 1, 64, 128, 8192, 128, 2, 8, FAKE, FAKE, FAKE, FAKE, 128, FAKE, FAKE,
                                  0.1, FAKE, 8192, 128, None, None, FAKE, 16, s) == L.EWORKSPACE
    # prompt beyond the limit
    assert lib.fastar_annca_select(FAKE, L.BF16, 1, 1, 64, 128, 8192, 128, FAKE, 2, FAKE, FAKE, 2000, 0.2, 16, 1,
                                   0, None, None, None, FAKE, FAKE, FAKE, FAKE, None, None, None, None, 0, s) == L.ECAPACITY
    # a bucket order needs the bucket count, and both of its arrays
    assert lib.fastar_annca_select(FAKE, L.BF16, 1, 1, 64, 128, 8192, 128, FAKE, 2, FAKE, FAKE, 100, 0.2, 16, 1,
                                   0, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, None, None, None, 0, s) == L.EINVAL
    assert lib.fastar_annca_select(FAKE, L.BF16, 1, 1, 64, 128, 8192, 128, FAKE, 2, FAKE, FAKE, 100, 0.2, 16, 1,
                                   8, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, None, None, None, None, 0, s) == L.EINVAL
    # kept-row planes: both or neither, with the values, bf16 only
    assert lib.fastar_annca_select(FAKE, L.BF16, 1, 1, 64, 128, 8192, 128, FAKE, 2, FAKE, FAKE, 100, 0.2, 16, 1,
                                   0, None, None, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 4096, None, None, 0,
                                   s) == L.EINVAL
    assert lib.fastar_annca_select(FAKE, L.BF16, 1, 1, 64, 128, 8192, 128, FAKE, 2, FAKE, FAKE, 100, 0.2, 16, 1,
                                   0, None, None, None, FAKE, FAKE, FAKE, FAKE, None, FAKE + 4096, FAKE + 8192, None, 0,
                                   s) == L.EINVAL
    assert lib.fastar_annca_select(FAKE, L.F32, 1, 1, 64, 128, 8192, 128, FAKE, 2, FAKE, FAKE, 100, 0.2, 16, 1,
                                   0, None, None, None, FAKE, FAKE, FAKE, FAKE, FAKE + 2048, FAKE + 4096, FAKE + 8192, None,
                                   0, s) == L.EUNSUPPORTED
    # the cross-attention over planes: bf16 planes, present and aligned
    assert lib.fastar_cross_attn_kept(FAKE, L.F32, 1, 1, 64, 128, 8192, 128, FAKE, FAKE, 100, FAKE, 0.1, FAKE, 8192,
                                      128, None, s) == L.EUNSUPPORTED
    assert lib.fastar_cross_attn_kept(FAKE, L.BF16, 1, 1, 64, 128, 8192, 128, None, FAKE, 100, FAKE, 0.1, FAKE, 8192,
                                      128, None, s) == L.EINVAL
    assert lib.fastar_cross_attn_kept(FAKE, L.BF16, 1, 1, 64, 128, 8192, 128, FAKE, FAKE + 8, 100, FAKE, 0.1, FAKE,
                                      8192, 128, None, s) == L.EINVAL
    # merge variant: the group counts are required, and compaction stays out-of-place for them too
    assert lib.fastar_cache_compact_merge(L.BF16, 1, 10, 128, 50, FAKE, FAKE, 1280, 128, FAKE, FAKE, FAKE,
                                          FAKE + 16, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE + 32, FAKE + 48,
                                          FAKE, FAKE, FAKE, FAKE, FAKE, None, s) == L.EINVAL
    assert lib.fastar_cache_compact_merge(L.BF16, 1, 10, 128, 50, FAKE, FAKE, 1280, 128, FAKE, FAKE, FAKE,
                                          FAKE + 16, FAKE, FAKE, FAKE + 64, FAKE, FAKE, FAKE, FAKE, FAKE + 32,
                                          FAKE + 48, FAKE + 4, FAKE + 8, FAKE + 64, FAKE, FAKE, None, s) == L.EINVAL
    assert lib.fastar_cache_compact_merge(L.BF16, 1, 100, 128, 50, FAKE, FAKE, 12800, 128, FAKE, FAKE, FAKE,
                                          FAKE + 16, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 32, FAKE + 48,
                                          FAKE, FAKE, FAKE, FAKE, FAKE, None, s) == L.ECAPACITY
    assert lib.fastar_sparse_attn_grouped(FAKE, L.BF16, 1, 64, 128, 8192, 128, 2, 8, FAKE, FAKE, FAKE, FAKE, 128,
                                          FAKE, FAKE, None, 0.1, FAKE, 8192, 128, None, None, FAKE, 1 << 30,
                                          s) == L.EINVAL
    assert lib.fastar_dense_attn_grouped(FAKE, L.BF16, 2, 64, 128, 8192, 128, FAKE, FAKE, 100, 12800, 128, FAKE, 50,
                                         0.1, FAKE, 8192, 128, None, s) == L.EINVAL
    # the sorted compaction needs its sorted copies, distinct from the caches, and a bucket count
    base = [L.BF16, 1, 10, 128, 50, FAKE, FAKE, 1280, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
            FAKE + 1024, FAKE + 2048, FAKE + 16, FAKE + 32, FAKE + 48, FAKE + 64]
    noq = [None, 0, None, None]   # no (query, slot) pair sort
    assert lib.fastar_cache_compact_sorted(*base, 8, FAKE, FAKE, FAKE, None, FAKE + 4096, *noq, None, s) == L.EINVAL
    assert lib.fastar_cache_compact_sorted(*base, 8, FAKE, FAKE, FAKE, FAKE + 8, FAKE + 4096, *noq, None,
                                           s) == L.EINVAL
    assert lib.fastar_cache_compact_sorted(*base, 8, FAKE, FAKE, FAKE, FAKE + 1024, FAKE + 4096, *noq, None,
                                           s) == L.EINVAL
    assert lib.fastar_cache_compact_sorted(*base, 0, FAKE, FAKE, FAKE, FAKE + 3072, FAKE + 4096, *noq, None,
                                           s) == L.EINVAL
    assert lib.fastar_cache_compact_sorted(*base, 300, FAKE, FAKE, FAKE, FAKE + 3072, FAKE + 4096, *noq, None,
                                           s) == L.ECAPACITY
    # with the pair sort: r in [1, FASTAR_MAX_R] and both outputs
    ok = [8, FAKE, FAKE, FAKE, FAKE + 3072, FAKE + 4096]
    assert lib.fastar_cache_compact_sorted(*base, *ok, FAKE, 0, FAKE, FAKE, None, s) == L.EINVAL
    assert lib.fastar_cache_compact_sorted(*base, *ok, FAKE, 2, None, FAKE, None, s) == L.EINVAL
    assert lib.fastar_cache_compact_sorted(*base, *ok, FAKE, 2, FAKE, None, None, s) == L.EINVAL
    assert lib.fastar_cache_compact_sorted(*base, *ok, FAKE, 99, FAKE, FAKE, None, s) == L.ECAPACITY
    # the presorted attention needs both sorted copies, 16-byte aligned
    assert lib.fastar_sparse_attn_presorted(FAKE, L.BF16, 1, 64, 128, 8192, 128, 2, 8, FAKE, FAKE, FAKE, FAKE,
                                            128, FAKE, FAKE, None, FAKE, 0.1, FAKE, 8192, 128, None, None, FAKE,
                                            1 << 30, s) == L.EINVAL
    assert lib.fastar_sparse_attn_presorted(FAKE, L.BF16, 1, 64, 128, 8192, 128, 2, 8, FAKE, FAKE, FAKE, FAKE,
                                            128, FAKE, FAKE, FAKE + 2, FAKE, 0.1, FAKE, 8192, 128, None, None,
                                            FAKE, 1 << 30, s) == L.EINVAL
    # the row kernels read their per-channel vectors 16 bytes at a time: misaligned ones are refused
    assert lib.fastar_layernorm_mod(FAKE, 1536, 10, 1536, 1e-6, None, None, FAKE + 4, None, None, None, FAKE,
                                    1536, s) == L.EINVAL
    assert lib.fastar_layernorm_mod(FAKE, 1536, 10, 1536, 1e-6, FAKE + 8, FAKE, None, None, None, None, FAKE,
                                    1536, s) == L.EINVAL
    assert lib.fastar_rmsnorm_rope(FAKE, 1536, 10, 1536, 128, 1e-6, FAKE + 4, 0, 0, None, 1, 1, 10000.0,
                                   s) == L.EINVAL
    # dense append past capacity
    assert lib.fastar_dense_append(L.BF16, 1, 64, 128, FAKE, FAKE, 8192, 128, FAKE, FAKE, 100, 50, s) == L.ECAPACITY
    # empty work is a successful no-op that touches nothing
    assert lib.fastar_bucket_assign(None, L.BF16, 4, 0, 128, 0, 128, None, 4, 1, None, None, None, s) == L.OK
    assert lib.fastar_dense_attn(None, L.BF16, 2, 0, 128, 0, 128, None, None, 0, 0, 128, 0.1, None, 0, 128, None,
                                 s) == L.OK


def test_binding_raises_on_error_code(lib):
    from kv_cache_tempcache_gb300 import _lib as L
    with pytest.raises(L.FastarError) as ei:
        L._call("fastar_dense_append", L.BF16, 1, 64, 128, FAKE, FAKE, 8192, 128, FAKE, FAKE, 100, 50, None)
    assert ei.value.code == L.ECAPACITY


def test_product_path_has_no_cpu_fallback():
    """The package never imports the oracle, and fails loudly without its library."""
    pkg = os.path.join(ROOT, "kv_cache_tempcache_gb300")
    for f in os.listdir(pkg):
        if f.endswith(".py"):
            src = open(os.path.join(pkg, f)).read()
            assert "from oracle" not in src and "import oracle" not in src, f
    from kv_cache_tempcache_gb300 import _lib
    with pytest.raises(FileNotFoundError):
        _lib.open_library("/nonexistent/libfastar.so")


def test_last_cuda_error_starts_clean(lib):
    # nothing has failed in this process: the CUDA-error diagnostic reports no error
    assert lib.fastar_last_cuda_error().decode() == "no error"


def _header_params():
    """name -> the C parameter types of every fastar_* declaration in the header."""
    out = {}
    for f in os.listdir(os.path.join(ROOT, "include")):
        if not f.endswith(".h"):
            continue
        text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", f)).read(), flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b(fastar_\w+)\s*\(([^)]*)\)\s*;", text):
            params = [p.strip() for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
            out[m.group(1)] = [re.sub(r"\s+\w+$", "", p) if "*" not in p else p for p in params]
    return out


def test_binding_signatures_match_the_header():
    # every declared parameter has a ctypes type of the same kind, in the same order
    from kv_cache_tempcache_gb300 import _lib
    kind = {"int": ctypes.c_int, "int64_t": ctypes.c_int64, "float": ctypes.c_float, "size_t": ctypes.c_size_t,
            "cudaStream_t": ctypes.c_void_p}
    decls = _header_params()
    assert len(decls) >= 12
    for name, params in decls.items():
        got = _lib._SIGS[name]
        want = [ctypes.c_void_p if "*" in p else kind[p.replace("const ", "").strip()] for p in params]
        assert got == want, f"{name}: binding {[t.__name__ for t in got]} vs header {params}"


def test_library_sources_call_no_allocator():
    # the library never allocates or frees device (or pinned host) memory: the caller owns
    # every buffer, and the allocation-free entry point relies on that for its whole path
    import os
    import re
    csrc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "kv_cache_tempcache_gb300", "csrc")
    pat = re.compile(r"\b(cudaMalloc\w*|cudaFree\w*|cudaHostAlloc|cudaMallocHost|cuMemAlloc\w*|cuMemCreate|"
                     r"cudaMemPoolCreate|malloc|calloc|realloc|new\s+\w)")
    hits = []
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            for n, line in enumerate(open(os.path.join(csrc, f)), 1):
                code = line.split("//")[0]
                if pat.search(code):
                    hits.append(f"{f}:{n}: {line.strip()}")
    assert not hits, "allocation calls in the library:\n" + "\n".join(hits)
