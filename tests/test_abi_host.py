"""Host side of the C ABI (no GPU): the library loads, exports every function
include/rvqmoe.h declares, computes sizes, and rejects bad arguments before
launching anything."""
import ctypes
import random

import pytest

import moe_expert_ffn_router_gb300 as rvq

lib = rvq._lib
A16 = 0x10000        # a fake, 16-byte aligned "device" address (never dereferenced)
A256 = 0x20000


def test_every_declared_function_is_exported():
    names = rvq.header_functions()
    assert len(names) >= 20
    missing = [n for n in names if not rvq.lib_has(n)]
    assert missing == []
    for n in ["rvq_pack", "rvq_lut_build", "rvq_gemv", "moe_route", "moe_expert_ffn",
              "moe_combine", "moe_layer_forward"]:
        assert n in names


def test_binding_constants_equal_the_header_defines():
    """Every numeric #define of include/rvqmoe.h that the binding also
    defines has the same value in both (the binding restates them)."""
    import re
    defines = {}
    for m in re.finditer(r"^#define\s+(\w+)\s+(0x[0-9a-fA-F]+|\d+)u?\b",
                         open(rvq.HEADER).read(), re.M):
        defines[m.group(1)] = int(m.group(2), 0)
    aliases = {"RVQ_DEV_ERR_INDEX": "DEV_ERR_INDEX", "RVQ_DEV_ERR_NONFINITE": "DEV_ERR_NONFINITE",
               "RVQ_DEV_ERR_CORRUPT": "DEV_ERR_CORRUPT", "RVQ_DEV_ERR_TIMEOUT": "DEV_ERR_TIMEOUT"}
    checked = 0
    for name, value in defines.items():
        py = getattr(rvq, aliases.get(name, name), None)
        if py is not None:
            assert py == value, (name, py, value)
            checked += 1
    assert checked >= 10, defines


def test_status_strings_and_version():
    for code in range(9):
        assert rvq.status_string(code) and rvq.status_string(code) != "unknown status"
    assert rvq.status_string(99) == "unknown status"
    assert rvq.rvq_version() == 0x000100


def test_code_bytes_is_exactly_three_bits_per_weight():
    assert rvq.rvq_code_bytes(32, 512) == 3 * 32 * 512 // 8
    assert rvq.rvq_code_bytes(2048, 7168) == 5_505_024
    assert rvq.rvq_code_bytes(7168, 2048) == 5_505_024
    for r, c in [(33, 512), (32, 500), (0, 512), (32, 0), (-32, 512)]:
        assert rvq.rvq_code_bytes(r, c) == 0


def test_bank_record_bytes():
    # header 128 + 3 packed codebooks + 3 matrices of 3*d*f/8, rounded to 256
    for d, f in [(2048, 1024), (7168, 2048), (512, 512)]:
        raw = 128 + 3 * 24576 + 3 * (3 * d * f // 8)
        assert rvq.moe_bank_record_bytes(d, f) == (raw + 255) // 256 * 256
    assert rvq.moe_bank_record_bytes(7168, 2048) == 16_589_056
    assert rvq.moe_bank_record_bytes(2000, 1024) == 0


def test_argument_checks_return_before_any_launch():
    s = None
    EINVAL, EALIGN, ENOMEM = 1, 2, 3
    assert lib.rvq_pack(A16, 33, 512, A16, 1 << 20, s) == EINVAL
    assert lib.rvq_pack(A16, 32, 512, A16 + 4, 1 << 20, s) == EALIGN
    assert lib.rvq_pack(A16, 32, 512, A16, 100, s) == ENOMEM
    assert lib.rvq_pack(None, 32, 512, A16, 1 << 20, s) == EINVAL
    assert lib.rvq_unpack(A16, 32, 512, A16, 100, s) == ENOMEM
    assert lib.rvq_lut_build(A16, A16, 0, 1, 12, A16, s) == EINVAL
    assert lib.rvq_lut_build(A16, A16, 7, 1, 16, A16, s) == EINVAL
    assert lib.rvq_gemv(A16, A16, 256, 512, A16 + 8, 0, 1, A16, A256, 1 << 20, s) == EALIGN
    assert lib.rvq_gemv(A16, A16, 256, 512, A16, 0, 1, A16, A256, 16, s) == ENOMEM
    assert lib.rvq_gemv(A16, A16, 256, 512, A16, 0, 0, A16, A256, 1 << 20, s) == EINVAL
    assert lib.moe_router_logits(A16, None, A16, 1, 1, 300, 512, A16, s) == EINVAL
    assert lib.moe_router_logits(A16, None, A16 + 2, 1, 1, 64, 512, A16, s) == EALIGN
    # routing: k > E, k > 32, n beyond the single-block limit, tiny workspace
    assert lib.moe_route(A16, 4, 8, 9, A16, A16, A16, A16, A256, 256, s) == EINVAL
    assert lib.moe_route(A16, 4, 64, 33, A16, A16, A16, A16, A256, 256, s) == EINVAL
    big = rvq.moe_route_max_tokens(256) + 1
    assert lib.moe_route(A16, big, 256, 16, A16, A16, A16, A16, A256, 256, s) == EINVAL
    assert lib.moe_route(A16, 4, 64, 8, A16, A16, A16, A16, A256, 8, s) == ENOMEM
    assert lib.moe_combine(A16, A16, 2, 2, 6, A16, 0, A16, s) == EINVAL
    assert lib.moe_combine(A16, A16, 2, 2, 8, A16, 1, A16, s) == EINVAL  # bf16 alias
    # offline encoder: too few or too many sub-vectors, ragged cols, bad iters,
    # unaligned workspace, short workspace
    ok = rvq.rvq_encode_workspace_bytes(256, 512)
    assert lib.rvq_encode(A16, 1, 2040, 2, A16, A16, A256, ok, s) == EINVAL      # N = 255
    assert lib.rvq_encode(A16, 2049, 8192, 2, A16, A16, A256, 1 << 40, s) == EINVAL  # N > 2^21
    assert lib.rvq_encode(A16, 256, 516, 2, A16, A16, A256, ok, s) == EINVAL
    assert lib.rvq_encode(A16, 256, 512, -1, A16, A16, A256, ok, s) == EINVAL
    assert lib.rvq_encode(A16, 256, 512, 2, A16, A16, A16 + 16, ok, s) == EINVAL
    assert lib.rvq_encode(A16, 256, 512, 2, A16, A16, A256, ok - 1, s) == ENOMEM
    assert lib.rvq_encode(None, 256, 512, 2, A16, A16, A256, ok, s) == EINVAL


def test_bank_init_checks():
    bank = rvq.RvqMoeBank()
    rb = rvq.moe_bank_record_bytes(2048, 1024)
    ok = lib.moe_bank_init(ctypes.byref(bank), A256, rb * 64, 64, 2048, 1024, 3)
    assert ok == 0 and bank.record_bytes == rb and bank.layer == 3 and bank.n_experts == 64
    assert lib.moe_bank_init(ctypes.byref(bank), A256 + 16, rb * 64, 64, 2048, 1024, 0) == 2
    assert lib.moe_bank_init(ctypes.byref(bank), A256, rb * 63, 64, 2048, 1024, 0) == 3
    assert lib.moe_bank_init(ctypes.byref(bank), A256, rb * 64, 0, 2048, 1024, 0) == 1
    assert lib.moe_bank_init(ctypes.byref(bank), A256, rb * 64, 64, 2000, 1024, 0) == 1
    assert b"multiples of 512" in lib.rvq_last_error()
    # a bank whose record size disagrees with its shape is refused
    bad = rvq.RvqMoeBank(A256, rb + 256, 64, 2048, 1024, 0)
    assert lib.moe_bank_validate(ctypes.byref(bad), None) == 1
    assert lib.moe_workspace_bytes(ctypes.byref(bank), 1, 8) > 256


def test_layer_graph_checks_before_capturing():
    """moe_layer_graph_create checks its arguments as the host-buffer layer
    call does, before any stream capture starts, and leaves *graph_out NULL;
    launching or destroying a NULL graph is refused / a no-op."""
    bank = rvq.RvqMoeBank()
    rb = rvq.moe_bank_record_bytes(2048, 1024)
    assert lib.moe_bank_init(ctypes.byref(bank), A256, rb * 64, 64, 2048, 1024, 0) == 0
    ws = lib.moe_workspace_bytes(ctypes.byref(bank), 4, 8)
    out = ctypes.c_void_p(12345)
    args = [ctypes.byref(bank), A16, None, None, 1, 4, 8, A16, A16, A16, A16, A16, A16, A16 + 0x100,
            None, A256, ws, 0, None, ctypes.byref(out)]
    def call(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        out.value = 12345
        rc = lib.moe_layer_graph_create(*a)
        assert out.value is None          # *graph_out cleared on every refusal
        return rc
    EINVAL, EALIGN, ENOMEM = 1, 2, 3
    assert lib.moe_layer_graph_create(*args[:-1], None) == EINVAL     # no graph_out
    assert call(a3=A16) == EINVAL                   # x_host without out_host
    assert call(a14=A16) == EINVAL                  # out_host without x_host
    assert call(a7=A16 + 2) == EALIGN               # x_dev
    assert call(a16=ws - 1) == ENOMEM               # workspace too small
    assert call(a5=0) == EINVAL                     # no tokens
    assert call(a4=7) == EINVAL                     # dtype
    assert call(a13=A16) == EINVAL                  # bf16 x aliasing out
    assert lib.moe_layer_graph_launch(None, None) == EINVAL
    assert lib.moe_layer_graph_destroy(None) == 0


def test_workspace_sizes_grow_with_batch():
    bank = rvq.RvqMoeBank()
    rb = rvq.moe_bank_record_bytes(7168, 2048)
    assert lib.moe_bank_init(ctypes.byref(bank), A256, rb * 256, 256, 7168, 2048, 0) == 0
    sizes = [lib.moe_workspace_bytes(ctypes.byref(bank), n, 16) for n in (1, 8, 64)]
    assert sizes[0] >= 256 + 16 * 2048 * 4  # at least h for 16 pairs
    assert sizes[0] < sizes[1] < sizes[2]
    assert lib.moe_workspace_bytes(None, 1, 16) == 0
    assert rvq.rvq_gemv_workspace_bytes(256, 512, 1) >= 256 + 256 * 4


def test_fuzz_argument_validation():
    """400 random argument sets (the pages report 400 fuzz cases for their own
    engine): every call returns a status; invalid shapes never return OK."""
    rng = random.Random(400)
    for _ in range(400):
        rows = rng.choice([0, 1, 31, 32, 64, 96, 2048, -32, 1 << 20])
        cols = rng.choice([0, 8, 256, 511, 512, 1024, 7168, -512])
        valid = rows > 0 and cols > 0 and rows % 32 == 0 and cols % 512 == 0
        rc = lib.rvq_pack(A16, rows, cols, A16 + rng.choice([0, 4]), 0, None)
        if not valid:
            assert rc == 1
        else:
            assert rc in (2, 3)  # misaligned or zero-byte destination, never launched
        n, E, k = rng.randint(-2, 5000), rng.randint(-2, 300), rng.randint(-2, 40)
        rc = lib.moe_route(A16, n, E, k, A16, A16, A16, A16, A256, 0, None)
        assert rc != 0


def test_encode_workspace_bytes():
    """Residual [N][8] fp32, assignment [N] int32, 256 x 8 int64 sums and 256
    int64 counts, each padded to 256 bytes; 0 for a shape the encoder refuses."""
    pad = lambda x: (x + 255) // 256 * 256
    for rows, cols in ((256, 512), (37, 72), (2048, 7168)):
        N = rows * cols // 8
        assert rvq.rvq_encode_workspace_bytes(rows, cols) == pad(32 * N) + pad(4 * N) + 16384 + 2048
    assert rvq.rvq_encode_workspace_bytes(1, 2040) == 0
    assert rvq.rvq_encode_workspace_bytes(2049, 8192) == 0
    assert rvq.rvq_encode_workspace_bytes(4, 500) == 0
