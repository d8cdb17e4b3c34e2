"""The C ABI without a GPU: the library builds and loads, exports every entry
point include/gdn.h declares, and rejects bad arguments on the host before
touching the device (these calls never reach the CUDA runtime)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._build_module().build()
    return ctypes.CDLL(path)


def test_header_declares_the_entry_points():
    names = set(_declared())
    assert {"gdn_gating", "causal_conv1d_fwd", "causal_conv1d_update", "gdn_prefill_chunked",
            "gdn_decode_recurrent", "gdn_state_snapshot", "gdn_get_device_status"} <= names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_lists_every_export(lib):
    import gated_deltanet_linear_10_gb300 as gdn
    assert set(gdn.EXPORTS) == set(_declared())


def test_status_strings_and_version(lib):
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_version.restype = ctypes.c_char_p
    assert lib.gdn_status_string(0) == b"GDN_OK"
    assert lib.gdn_status_string(1) == b"GDN_ERR_INVALID_ARG"
    assert lib.gdn_status_string(2) == b"GDN_ERR_UNSUPPORTED"
    assert lib.gdn_status_string(99) == b"GDN_STATUS_UNKNOWN"
    assert b"sm_103a" in lib.gdn_version()


V, I32, I64, F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
FAKE = V(0x1000)   # never dereferenced: every call below fails its host check first


def test_host_argument_checks(lib):
    # gating: null outputs / bad dtype / negative sizes
    f = lib.gdn_gating
    f.argtypes = [V, V, V, V, I64, I32, I32, V, V, V]
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 2, 1, None, FAKE, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 2, 7, FAKE, FAKE, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, -1, 2, 1, FAKE, FAKE, None) == 1
    assert f(None, None, None, None, 0, 2, 1, None, None, None) == 0     # empty: no launch
    # decode: unsupported head size, hv not a multiple of hqk, too many tokens
    d = lib.gdn_decode_recurrent
    d.argtypes = [V, I64, V, I64, V, I64, V, V, I32, I32, I32, I32, I32, I32, F32, I32, V, I64,
                  V, V, V, I32, V]
    args = lambda tps, hqk, hv, dk, dv: (FAKE, 2048, FAKE, 2048, FAKE, 4096, FAKE, FAKE, 4, tps,
                                         hqk, hv, dk, dv, 1.0, 1, FAKE, 8, FAKE, None, FAKE, 1,
                                         None)
    assert d(*args(1, 16, 32, 96, 128)) == 2
    assert d(*args(1, 16, 24, 128, 128)) == 1
    assert d(*args(17, 16, 32, 128, 128)) == 2
    # prefill: dk != dv, unsupported chunk
    p = lib.gdn_prefill_chunked
    p.argtypes = [V, I64, V, I64, V, I64, V, V, V, I32, I64, I32, I32, I32, I32, F32, I32, I32, V,
                  I64, V, V, V, I32, V, ctypes.c_size_t, V]
    base = [FAKE, 2048, FAKE, 2048, FAKE, 4096, FAKE, FAKE, FAKE, 2, 100, 16, 32, 128, 128, 1.0, 1,
            64, FAKE, 8, FAKE, FAKE, FAKE, 1, None, 0, None]
    bad = list(base); bad[14] = 64
    assert p(*bad) == 2
    bad = list(base); bad[17] = 48
    assert p(*bad) == 2
    bad = list(base); bad[1] = 100      # row stride shorter than hqk*dk
    assert p(*bad) == 1
    # conv: width 5 unsupported, channels not a multiple of 8
    c = lib.causal_conv1d_update
    c.argtypes = [V, I32, I32, I32, I32, V, V, V, I64, V, V, I32, V, I32, V]
    assert c(FAKE, 4, 1, 8192, 5, FAKE, None, FAKE, 8, FAKE, None, 1, FAKE, 1, None) == 2
    assert c(FAKE, 4, 1, 8190, 4, FAKE, None, FAKE, 8, FAKE, None, 1, FAKE, 1, None) == 2
    # snapshot: slot size not a multiple of 16 bytes
    s = lib.gdn_state_snapshot
    s.argtypes = [V, I64, I64, V, V, I32, V]
    assert s(FAKE, 8, 24, FAKE, FAKE, 2, None) == 1
    assert s(FAKE, 8, 32, FAKE, FAKE, 0, None) == 0


def test_mixed_batch_host_checks(lib):
    """n_decode outside 0 .. n_seqs, decode rows without initial slots, and an
    unsupported head size in the decode half fail before anything launches."""
    m = lib.gdn_mixed_batch
    m.argtypes = [V, I64, V, I64, V, I64, V, V, V, I32, I32, I64, I32, I32, I32, I32, F32, I32,
                  I32, V, I64, V, V, I32, V, I32, V, ctypes.c_size_t, V]
    base = [FAKE, 2048, FAKE, 2048, FAKE, 4096, FAKE, FAKE, FAKE, 4, 2, 100, 16, 32, 128, 128,
            1.0, 1, 64, FAKE, 8, FAKE, FAKE, 1, FAKE, 1, None, 0, None]
    bad = list(base); bad[10] = 5        # n_decode > n_seqs
    assert m(*bad) == 1
    bad = list(base); bad[10] = -1
    assert m(*bad) == 1
    bad = list(base); bad[11] = 1        # fewer tokens than decode rows
    assert m(*bad) == 1
    bad = list(base); bad[21] = None     # decode rows need their initial slots
    assert m(*bad) == 1
    bad = list(base); bad[22] = None; bad[23] = 0   # ... and final slots unless in place
    assert m(*bad) == 1
    bad = list(base); bad[14] = 96       # dk 96: the decode half is unsupported
    bad[15] = 96
    assert m(*bad) == 2
    # a valid decode half with a prefill half that fails its checks: neither
    # launches (a launch here, with no GPU, would return GDN_ERR_LAUNCH)
    bad = list(base); bad[18] = 48       # chunk 48: the prefill half is unsupported
    assert m(*bad) == 2
    empty = list(base); empty[9] = 0; empty[10] = 0; empty[11] = 0
    assert m(*empty) == 0                # nothing to do: no launch


def test_prefill_workspace_size(lib):
    """Only the bf16 dk = dv = 128, chunk-64 path uses scratch: a small header
    plus one operand block per (chunk bound, V head) item, where the chunk
    bound is ceil(n_tokens / 64) + n_seqs."""
    f = lib.gdn_prefill_workspace_size
    f.argtypes = [I32, I64, I32, I32, I32, I32, I32]
    f.restype = ctypes.c_size_t
    F32_, BF16_ = 0, 1
    assert f(4, 1000, 32, 64, 64, 64, BF16_) == 0
    assert f(4, 1000, 32, 128, 128, 64, F32_) == 0
    assert f(4, 1000, 32, 128, 128, 32, BF16_) == 0
    assert f(4, 0, 32, 128, 128, 64, BF16_) == 0
    a = f(4, 1000, 32, 128, 128, 64, BF16_)          # bound 16 + 4
    b = f(4, 1024, 32, 128, 128, 64, BF16_)          # same bound
    c = f(4, 1025, 32, 128, 128, 64, BF16_)          # bound 17 + 4
    assert a > 0 and a == b
    item = (c - a) // 32
    assert c - a == 32 * item and item >= 3 * 64 * 128   # at least T1, T2, P in bf16
    assert a - 20 * 32 * item in (1024, 2048)          # header: n_seqs + 1 offsets, 1 KiB pages


def test_gated_rmsnorm_host_checks(lib):
    """Unsupported head size, misaligned z or stride, negative eps: refused
    on the host before any launch."""
    f = lib.gdn_gated_rmsnorm
    f.argtypes = [V, V, I64, V, I64, I32, I32, F32, V, I32, V]
    A = 1 << 20                                   # 16-byte aligned fake addresses
    assert f(A, A, 512, A, 4, 4, 96, 1e-6, A, 1, None) == 2        # dv 96 not built
    assert f(A, A + 2, 512, A, 4, 4, 128, 1e-6, A, 1, None) == 1    # z not 4-element aligned
    assert f(A, A, 514, A, 4, 4, 128, 1e-6, A, 1, None) == 1        # stride not a multiple of 4
    assert f(A, A, 512, A, 4, 4, 128, -1.0, A, 1, None) == 1        # eps < 0
    assert f(A, A, 256, A, 4, 4, 128, 1e-6, A, 1, None) == 1        # stride < hv * dv
    assert f(None, None, 512, None, 0, 4, 128, 1e-6, None, 1, None) == 0   # empty: no launch


def test_gated_prefill_host_checks(lib):
    """The gated prefill runs the prefill's and the norm's host checks before
    any launch: a bad prefill shape, a missing or misaligned z, a z row stride
    shorter than a token, a negative eps and a missing weight are refused."""
    f = lib.gdn_prefill_chunked_gated
    f.argtypes = [V, I64, V, I64, V, I64, V, V, V, I32, I64, I32, I32, I32, I32, F32, I32, I32,
                  V, I64, V, V, V, I64, V, F32, V, I32, V, ctypes.c_size_t, V]
    A = 1 << 20
    base = [A, 2048, A, 2048, A, 4096, A, A, A, 2, 100, 16, 32, 128, 128, 1.0, 1, 64, A, 8, A, A,
            A, 4096, A, 1e-6, A, 1, None, 0, None]
    bad = list(base); bad[17] = 48          # chunk 48: the prefill is not built
    assert f(*bad) == 2
    bad = list(base); bad[22] = None        # no z
    assert f(*bad) == 1
    bad = list(base); bad[22] = A + 2       # z not 4-element aligned
    assert f(*bad) == 1
    bad = list(base); bad[23] = 4000        # z row stride < hv * dv
    assert f(*bad) == 1
    bad = list(base); bad[25] = -1.0        # eps < 0
    assert f(*bad) == 1
    bad = list(base); bad[24] = None        # no norm weight
    assert f(*bad) == 1


def test_fused_step_host_checks(lib):
    """The fused decode and MTP steps refuse bad shapes and pointers on the
    host: unsupported V heads per QK head, tokens per sequence outside 1..16,
    a row stride shorter than a row, missing buffers, a misaligned pool; an
    empty batch launches nothing.  The decode step's workspace size is y
    (bf16) plus g and beta (fp32), each rounded up to 256 bytes."""
    ws = lib.gdn_decode_step_workspace_size
    ws.argtypes = [I32, I32, I32]
    ws.restype = ctypes.c_size_t
    assert ws(256, 16, 32) == 256 * 8192 * 2 + 2 * 256 * 32 * 4
    assert ws(3, 1, 2) == 3 * 512 * 2 + 2 * 256
    assert ws(0, 16, 32) == 0
    d = lib.gdn_decode_step_fused
    d.argtypes = [V, I64, V, V, V, V, V, V, V, I32, I32, I32, F32, V, I64, V, V, ctypes.c_size_t,
                  V, V]
    A = 1 << 20
    base = [A, 8192, A, None, A, A, A, A, A, 4, 16, 32, 1.0, A, 8, A, None, 0, A, None]
    bad = list(base); bad[10] = 8           # 4 V heads per QK head
    assert d(*bad) == 2
    bad = list(base); bad[1] = 8000         # row stride < channels
    assert d(*bad) == 1
    bad = list(base); bad[18] = None        # no o
    assert d(*bad) == 1
    bad = list(base); bad[9] = 0            # empty: no launch
    assert d(*bad) == 0
    m = lib.gdn_mtp_step_fused
    m.argtypes = [V, I64, V, V, V, V, V, V, V, I32, I32, I32, I32, F32, V, I64, V, V, V, V]
    base = [A, 8192, A, None, A, A, A, A, A, 4, 4, 16, 32, 1.0, A, 8, A, A, A, None]
    bad = list(base); bad[10] = 17          # 17 tokens per sequence
    assert m(*bad) == 2
    bad = list(base); bad[10] = 0
    assert m(*bad) == 2
    bad = list(base); bad[12] = 24          # hv not a multiple of hqk
    assert m(*bad) == 1
    bad = list(base); bad[17] = None        # snapshots are required
    assert m(*bad) == 1
    bad = list(base); bad[1] = 4096         # row stride < channels
    assert m(*bad) == 1
    bad = list(base); bad[4] = A + 8        # conv state pool not 16-byte aligned
    assert m(*bad) == 1
    bad = list(base); bad[9] = 0            # empty: no launch
    assert m(*bad) == 0


def test_prefill_layer_host_checks(lib):
    """The one-call prefill layer refuses, before any launch: hv not a
    multiple of hqk, missing raw gates, a workspace below its size or not
    1 KiB aligned, an unaligned o; an empty batch launches nothing.  Its
    workspace size is y (bf16, rounded up to 1 KiB) plus the prefill's."""
    ws = lib.gdn_prefill_layer_workspace_size
    ws.argtypes = [I32, I64, I32, I32]
    ws.restype = ctypes.c_size_t
    pws = lib.gdn_prefill_workspace_size
    pws.argtypes = [I32, I64, I32, I32, I32, I32, I32]
    pws.restype = ctypes.c_size_t
    assert ws(8, 20668, 16, 32) == (20668 * 8192 * 2 + 1023) // 1024 * 1024 + \
        pws(8, 20668, 32, 128, 128, 64, 1)
    assert ws(0, 100, 16, 32) == 0
    f = lib.gdn_prefill_layer
    f.argtypes = [V, I64, V, V, V, I64, V, V, V, V, V, V, V, I32, I64, I32, I32, F32, V, I64, V, V,
                  V, V, ctypes.c_size_t, V]
    A = 1 << 20
    need = ws(2, 100, 2, 4)
    base = [A, 1024, A, None, A, 8, A, None, A, A, A, A, A, 2, 100, 2, 4, 1.0, A, 8, A, A, A, A,
            need, None]
    bad = list(base); bad[16] = 5           # hv not a multiple of hqk
    assert f(*bad) == 1
    bad = list(base); bad[8] = None         # no raw a
    assert f(*bad) == 1
    bad = list(base); bad[24] = need - 1    # workspace too small
    assert f(*bad) == 1
    bad = list(base); bad[23] = A + 512     # workspace not 1 KiB aligned
    assert f(*bad) == 1
    bad = list(base); bad[22] = A + 8       # o not 16-byte aligned
    assert f(*bad) == 1
    bad = list(base); bad[13] = 0; bad[14] = 0   # empty: no launch
    assert f(*bad) == 0


def test_prefill_layer_gated_host_checks(lib):
    """The gated layer call refuses, before any launch, what the plain one
    refuses, and also: no z, a z row stride below hv * 128 or not a multiple
    of 4, no norm weight, a negative eps; an empty batch launches nothing."""
    ws = lib.gdn_prefill_layer_workspace_size
    ws.argtypes = [I32, I64, I32, I32]
    ws.restype = ctypes.c_size_t
    f = lib.gdn_prefill_layer_gated
    f.argtypes = [V, I64, V, V, V, I64, V, V, V, V, V, V, V, I32, I64, I32, I32, F32, V, I64, V, V,
                  V, I64, V, F32, V, V, ctypes.c_size_t, V]
    A = 1 << 20
    need = ws(2, 100, 2, 4)
    base = [A, 1024, A, None, A, 8, A, None, A, A, A, A, A, 2, 100, 2, 4, 1.0, A, 8, A, A,
            A, 4 * 128, A, 1e-6, A, A, need, None]
    bad = list(base); bad[16] = 5           # hv not a multiple of hqk
    assert f(*bad) == 1
    bad = list(base); bad[22] = None        # no z
    assert f(*bad) == 1
    bad = list(base); bad[23] = 4 * 128 - 4  # z rows shorter than hv * 128
    assert f(*bad) == 1
    bad = list(base); bad[23] = 4 * 128 + 2  # z row stride not a multiple of 4
    assert f(*bad) == 1
    bad = list(base); bad[24] = None        # no norm weight
    assert f(*bad) == 1
    bad = list(base); bad[25] = -1.0        # negative eps
    assert f(*bad) == 1
    bad = list(base); bad[28] = need - 1    # workspace too small
    assert f(*bad) == 1
    bad = list(base); bad[26] = A + 8       # y not 16-byte aligned
    assert f(*bad) == 1
    bad = list(base); bad[13] = 0; bad[14] = 0   # empty: no launch
    assert f(*bad) == 0
