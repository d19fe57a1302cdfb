"""C-ABI checks that need no GPU: the library builds and loads, exports every
entry point declared in include/fp8q.h, and rejects bad arguments on the host
before anything touches CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8q.h")

FAKE = 1 << 20  # a non-NULL, 16-byte-aligned pointer value that is never dereferenced


@pytest.fixture(scope="module")
def L():
    from scaling_quantization_gemm_gb300 import build as b
    b.build()
    import scaling_quantization_gemm_gb300 as q
    return q.lib()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    syms = declared_symbols()
    for s in ["fp8_amax", "fp8_compute_scale", "fp8_amax_history_update", "fp8_quantize", "fp8_quantize_current",
              "fp8_scaled_gemm"]:
        assert s in syms


def test_library_exports_every_declared_symbol(L):
    for s in declared_symbols():
        assert hasattr(L, s), s
    import scaling_quantization_gemm_gb300 as q
    assert set(q.ENTRY_POINTS) <= set(declared_symbols())


def test_library_exports_nothing_else(L):
    # the shared object is built with hidden visibility: only the C ABI is exported
    out = os.popen(f"nm -D --defined-only {L._name}").read()
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert {s for s in exported if s.startswith("fp8_")} == set(declared_symbols())


def test_status_strings(L):
    import scaling_quantization_gemm_gb300 as q
    assert [q.status_name(i) for i in range(5)] == ["FP8_OK", "FP8_ERR_INVALID_ARG", "FP8_ERR_UNSUPPORTED",
                                                    "FP8_ERR_CUDA", "FP8_ERR_TIMEOUT"]


def _detail(L):
    return L.fp8_last_error_detail().decode()


def test_amax_validation(L):
    assert L.fp8_amax(None, 4, 8, 8, FAKE, None) == 1
    assert L.fp8_amax(FAKE, -1, 8, 8, FAKE, None) == 1
    assert L.fp8_amax(FAKE, 4, 8, 4, FAKE, None) == 1  # ld < cols
    assert L.fp8_amax(FAKE, 4, 8, 8, None, None) == 1
    assert L.fp8_amax(FAKE, 4, 12, 12, FAKE, None) == 2  # cols % 8
    assert L.fp8_amax(FAKE + 2, 4, 8, 8, FAKE, None) == 2  # misaligned
    assert "aligned" in _detail(L)
    assert L.fp8_amax(FAKE, 0, 8, 8, FAKE, None) == 0  # empty: valid no-op


def test_compute_scale_and_history_validation(L):
    assert L.fp8_compute_scale(None, 0, 0, FAKE, FAKE, FAKE, None, None) == 1
    assert L.fp8_compute_scale(FAKE, 7, 0, FAKE, FAKE, FAKE, None, None) == 1
    assert L.fp8_compute_scale(FAKE, 0, 0, None, None, None, None, None) == 1
    h = [FAKE] * 3
    assert L.fp8_amax_history_update(FAKE, 0, FAKE, FAKE, 0, 0, *h, None, None) == 1
    assert L.fp8_amax_history_update(FAKE, 70000, FAKE, FAKE, 0, 0, *h, None, None) == 1
    assert L.fp8_amax_history_update(FAKE, 16, None, FAKE, 0, 0, *h, None, None) == 1
    assert L.fp8_amax_history_update(FAKE, 16, FAKE + 4, FAKE, 0, 0, *h, None, None) == 1


def test_quantize_validation(L):
    q = L.fp8_quantize
    # per-tensor needs scale, takes no block scales
    assert q(FAKE, 32, 32, 32, 0, 0, 0, None, FAKE, None, None, None, None, None) == 1
    assert q(FAKE, 32, 32, 32, 0, 0, 0, FAKE, FAKE, None, FAKE, None, None, None) == 1
    # no outputs
    assert q(FAKE, 32, 32, 32, 0, 0, 0, FAKE, None, None, None, None, None, None) == 1
    # block: needs matching scale tensors, no per-tensor scale
    assert q(FAKE, 32, 32, 32, 0, 3, 0, None, FAKE, None, None, None, None, None) == 1
    assert q(FAKE, 32, 32, 32, 0, 3, 0, FAKE, FAKE, None, FAKE, None, None, None) == 1
    assert q(FAKE, 32, 32, 32, 0, 1, 0, None, FAKE, FAKE, FAKE, None, None, None) == 1  # q_col without sf_col
    # bad enums
    assert q(FAKE, 32, 32, 32, 2, 0, 0, FAKE, FAKE, None, None, None, None, None) == 1
    assert q(FAKE, 32, 32, 32, 0, 9, 0, FAKE, FAKE, None, None, None, None, None) == 1
    # column-wise output needs rows % 16 == 0
    assert q(FAKE, 24, 32, 32, 0, 0, 0, FAKE, None, FAKE, None, None, None, None) == 2
    # empty is a no-op
    assert q(FAKE, 0, 32, 32, 0, 0, 0, FAKE, FAKE, None, None, None, None, None) == 0


def test_gemm_validation(L):
    g = L.fp8_scaled_gemm
    args = lambda **kw: [kw.get("op", 0), kw.get("M", 128), kw.get("N", 256), kw.get("K", 128), FAKE,
                         kw.get("lda", 128), 0, kw.get("ga", 0), FAKE, FAKE, kw.get("ldb", 128), 0, kw.get("gb", 0),
                         FAKE, FAKE, kw.get("out", 0), kw.get("ldd", 256), None, None]
    assert g(*args(op=5)) == 1
    assert g(*args(M=-1)) == 1
    assert g(*args(ga=0, gb=3)) == 1  # per-tensor on one side only
    assert g(*args(ldd=128)) == 1
    assert g(*args(K=120, lda=128, ldb=128)) == 2  # K % 16
    assert g(*args(N=200, ldd=256)) == 2  # N % 16
    assert g(*args(ga=3, gb=3, K=160, lda=160, ldb=160)) == 2  # block-scaled needs K % 128
    assert g(*args(lda=64)) == 1  # lda < K
    assert g(*args(M=0)) == 0  # empty output: no-op


def test_quantize_batch_validation(L):
    """fp8_quantize_batch: the descriptor layout (96 bytes), n in [0, 4], reserved = 0, and every
    descriptor checked as fp8_quantize checks its arguments before anything is launched; the error
    detail names the descriptor."""
    import scaling_quantization_gemm_gb300 as q
    assert ctypes.sizeof(q.QuantizeDesc) == 96 and q.QUANTIZE_BATCH_MAX == 4
    text = open(HEADER).read()
    assert re.search(r"#define FP8_QUANTIZE_BATCH_MAX (\d+)", text).group(1) == "4"
    f = L.fp8_quantize_batch
    assert f(None, 0, None) == 0  # empty: no-op
    assert f(None, -1, None) == 1 and f(None, 5, None) == 1
    assert f(None, 2, None) == 1  # NULL descriptors
    descs = (q.QuantizeDesc * 3)()
    for d in descs:
        d.x, d.rows, d.cols, d.ld, d.fmt, d.gran = FAKE, 32, 64, 64, 0, 3
        d.q_row, d.sf_row = FAKE, FAKE
    descs[0].gran, descs[0].sf_row, descs[0].scale = 0, None, FAKE  # per-tensor
    addr = ctypes.cast(descs, ctypes.c_void_p)
    # descriptor 2 invalid in turn: rejected before any launch, detail names it
    for field, bad, good, code in (("reserved", 1, 0, 1), ("fmt", 4, 0, 1), ("gran", 9, 3, 1), ("ld", 32, 64, 1),
                                   ("cols", 60, 64, 2), ("x", FAKE + 8, FAKE, 2), ("sf_row", None, FAKE, 1),
                                   ("q_row", FAKE + 4, FAKE, 2), ("rows", -1, 32, 1)):
        setattr(descs[2], field, bad)
        assert f(addr, 3, None) == code, field
        assert _detail(L).startswith("descriptor 2:"), (field, _detail(L))
        setattr(descs[2], field, good)
    descs[1].scale = FAKE  # a block cast given a per-tensor scale
    assert f(addr, 3, None) == 1 and _detail(L).startswith("descriptor 1:")


def test_block_scaled_k_rule_matches_the_header(L):
    """The header states that every block-scaled mode needs K % 128 == 0; the check returns
    FP8_ERR_UNSUPPORTED for K = 32, 64, 96 and 160 in each mode (MX 1x32 included)."""
    text = " ".join(w for line in open(HEADER) for w in line.strip().lstrip("*").split())
    assert "Every block-scaled mode (1x128, 128x128 and MX 1x32 alike) needs K % 128 == 0" in text
    g = L.fp8_scaled_gemm
    for ga, gb in ((3, 3), (1, 2), (1, 1), (2, 2), (4, 4)):
        for K in (32, 64, 96, 160):
            assert g(0, 256, 256, K, FAKE, 256, 0, ga, FAKE, FAKE, 256, 0, gb, FAKE, FAKE, 1, 256, None, None) == 2


def test_quantize_current_validation(L):
    qc = L.fp8_quantize_current
    a = lambda **kw: [kw.get("x", FAKE), kw.get("rows", 32), kw.get("cols", 32), kw.get("ld", 32), kw.get("fmt", 0),
                      0, kw.get("q_row", FAKE), kw.get("q_col", None), FAKE, FAKE, FAKE, FAKE, kw.get("ws", FAKE),
                      None, None]
    assert qc(*a(ws=None)) == 1
    assert "workspace" in _detail(L)
    assert qc(*a(ws=FAKE + 8)) == 1  # workspace not 16-byte aligned
    assert qc(*a(fmt=3)) == 1
    assert qc(*a(q_row=None)) == 1  # no output
    assert qc(*a(ld=16)) == 1  # ld < cols
    assert qc(*a(cols=12, ld=12)) == 2
    assert qc(*a(rows=24, q_col=FAKE)) == 2  # column-wise output needs rows % 16


def test_workspace_size_constant_matches_header(L):
    import scaling_quantization_gemm_gb300 as q
    text = open(HEADER).read()
    m = re.search(r"#define FP8_QUANTIZE_CURRENT_WORKSPACE_BYTES (\d+)", text)
    assert m and int(m.group(1)) == q.QUANTIZE_CURRENT_WORKSPACE_BYTES


def test_quantize_current_noalloc_validation(L):
    qn = L.fp8_quantize_current_noalloc
    a = lambda **kw: [kw.get("x", FAKE), kw.get("rows", 32), kw.get("cols", 32), kw.get("ld", 32), kw.get("fmt", 0),
                      0, kw.get("q_row", FAKE), kw.get("q_col", None), FAKE, FAKE, FAKE, FAKE, None, None]
    assert qn(*a(fmt=3)) == 1
    assert qn(*a(q_row=None)) == 1
    assert qn(*a(x=None)) == 1
    assert qn(*a(ld=16)) == 1
    assert qn(*a(cols=12, ld=12)) == 2
    assert qn(*a(rows=24, q_col=FAKE)) == 2


def test_gemm_quantize_validation(L):
    g = L.fp8_scaled_gemm_quantize
    args = lambda **kw: [kw.get("op", 0), kw.get("M", 128), kw.get("N", 256), kw.get("K", 128), FAKE,
                         kw.get("lda", 128), 0, FAKE, FAKE, kw.get("ldb", 128), 0, FAKE, kw.get("Dq", FAKE),
                         kw.get("ldd", 256), kw.get("fd", 0), kw.get("sd", FAKE), None, None, None]
    assert g(*args(op=4)) == 1
    assert g(*args(fd=5)) == 1
    assert g(*args(sd=None)) == 1
    assert g(*args(Dq=None)) == 1
    assert g(*args(ldd=200)) == 1  # ldd < N
    assert g(*args(N=200, ldd=256)) == 2  # N % 16
    assert g(*args(Dq=FAKE + 8)) == 2  # Dq alignment
    assert g(*args(K=120, lda=128, ldb=128)) == 2
    assert g(*args(M=0)) == 0


def test_set_bias_and_cast_stats_validation(L):
    assert L.fp8_set_bias(128, FAKE, FAKE, FAKE, None) == 1
    assert L.fp8_set_bias(-127, FAKE, FAKE, FAKE, None) == 1
    assert L.fp8_set_bias(0, None, None, None, None) == 1
    cs = L.fp8_cast_stats
    assert cs(FAKE, 32, 32, 32, 0, FAKE, 0, FAKE, FAKE, None) == 1  # n = 0
    assert cs(FAKE, 32, 32, 32, 0, FAKE, 9, FAKE, FAKE, None) == 1  # n > 8
    assert cs(FAKE, 32, 32, 32, 2, FAKE, 1, FAKE, FAKE, None) == 1  # format
    assert cs(FAKE, 32, 32, 32, 0, FAKE, 1, None, FAKE, None) == 1
    assert cs(FAKE, 32, 32, 32, 0, FAKE, 1, FAKE + 4, FAKE, None) == 1  # counters 8-byte aligned
    assert cs(FAKE, 32, 12, 12, 0, FAKE, 1, FAKE, FAKE, None) == 2  # cols % 8
    assert cs(FAKE, 0, 32, 32, 0, FAKE, 1, FAKE, FAKE, None) == 0  # empty


def test_compute_scale_ratio_validation(L):
    assert L.fp8_compute_scale_ratio(None, 0, FAKE, FAKE, None, None) == 1
    assert L.fp8_compute_scale_ratio(FAKE, 3, FAKE, FAKE, None, None) == 1
    assert L.fp8_compute_scale_ratio(FAKE, 0, None, None, None, None) == 1
    q = L.fp8_quantize
    assert q(FAKE, 32, 32, 32, 0, 5, 0, None, FAKE, None, FAKE, None, None, None) == 1  # granularity 5 unknown


def test_quantize_f32_validation(L):
    f = L.fp8_quantize_f32
    assert f(None, 0, 0, None, None, None, None) == 0          # empty: no-op, nothing required
    assert f(FAKE, -1, 0, None, FAKE, None, None) == 1         # negative size
    assert f(FAKE, 8, 2, None, FAKE, None, None) == 1          # unknown format
    assert f(None, 8, 0, None, FAKE, None, None) == 1          # x required
    assert f(FAKE, 8, 0, None, None, None, None) == 1          # q required
    assert f(FAKE + 4, 8, 0, None, FAKE, None, None) == 2      # x not 16-byte aligned
    assert f(FAKE, 8, 0, None, FAKE + 2, None, None) == 2      # q not 8-byte aligned
    assert f(FAKE, 8, 0, FAKE + 1, FAKE, None, None) == 1      # scale misaligned


def test_cast_dimensions_past_2_31_rejected(L):
    big = 1 << 31
    # fp8_quantize / fp8_quantize_current / _noalloc: TMA coordinates are 32-bit
    assert L.fp8_quantize(FAKE, big, 8, 8, 0, 0, 0, FAKE, FAKE, None, None, None, None, None) == 2
    assert L.fp8_quantize(FAKE, 8, big, big, 0, 0, 0, FAKE, FAKE, None, None, None, None, None) == 2
    assert L.fp8_quantize_current(FAKE, big, 8, 8, 0, 0, FAKE, None, None, None, None, None, FAKE, None, None) == 2
    assert L.fp8_quantize_current_noalloc(FAKE, 8, big, big, 0, 0, FAKE, None, None, None, None, None, None,
                                          None) == 2


def test_history_batch_validation(L):
    import scaling_quantization_gemm_gb300 as q
    assert ctypes.sizeof(q.HistoryStateRecord) == 72  # fp8_history_state
    f = L.fp8_amax_history_update_batch
    assert f(None, 0, None) == 0  # empty: no-op
    assert f(None, -1, None) == 1
    assert f(None, 2, None) == 1
    recs = (q.HistoryStateRecord * 2)()
    for r in recs:
        r.history = r.pos = r.amax = r.bias = r.scale = r.scale_inv = FAKE
        r.len, r.fmt = 16, 0
    addr = ctypes.cast(recs, ctypes.c_void_p)
    # record 1 invalid in turn: rejected before any launch
    for field, bad, good in (("len", 0, 16), ("len", 65537, 16), ("fmt", 7, 1), ("reserved", 3, 0),
                             ("pos", FAKE + 4, FAKE), ("status", FAKE + 2, None), ("scale", None, FAKE)):
        setattr(recs[1], field, bad)
        assert f(addr, 2, None) == 1, field
        setattr(recs[1], field, good)


def test_binding_argument_counts_match_the_header(L):
    """Every entry point's ctypes argument list has as many entries as its declaration has
    parameters (the binding and the header cannot drift apart unnoticed)."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    decls = dict(re.findall(r"FP8Q_API\s+[^;(]*?\b(fp8_[a-z_0-9]+)\s*\(([^)]*)\)\s*;", text))
    import scaling_quantization_gemm_gb300 as q
    q.lib()
    checked = 0
    for name in q.ENTRY_POINTS:
        params = decls[name].strip()
        n = 0 if params in ("", "void") else params.count(",") + 1
        argtypes = getattr(L, name).argtypes
        if argtypes is None:
            continue
        assert len(argtypes) == n, (name, len(argtypes), n)
        checked += 1
    assert checked >= 12
