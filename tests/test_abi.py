"""The C-ABI library builds, loads without a GPU and exports every symbol the
header declares; host-side validation rejects bad arguments before any CUDA
call.  No compute runs here."""
import ctypes
import os
import re
import subprocess

import pytest

import paged_kv_cache_156_gb300 as pkv
from paged_kv_cache_156_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert declared_symbols() == sorted(pkv.ABI_SYMBOLS)


def test_header_constants_match_the_binding():
    """The values the header defines and the binding passes (PKV_PLANNED, PKV_INPUTS_READY,
    PKV_PLAN_MAX_SEQS) agree."""
    text = open(HEADER).read()
    defined = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define\s+(PKV_\w+)\s+(\d+)\s*$", text, re.M)}
    assert defined["PKV_PLANNED"] == pkv.PLANNED
    assert defined["PKV_INPUTS_READY"] == pkv.INPUTS_READY
    assert defined["PKV_PLAN_MAX_SEQS"] == pkv.PLAN_MAX_SEQS
    assert pkv.PLANNED & pkv.INPUTS_READY == 0


def _c_kind(decl):
    """A C parameter or return type from the header, reduced to what ctypes must pass."""
    decl = re.sub(r"\b(const|struct)\b", " ", decl)
    if "*" in decl:
        return "char_p" if re.fullmatch(r"\s*char\s*\*\s*", decl) else "ptr"
    t = decl.split()[0] if decl.split() else "void"
    return {"int": "int", "pkv_dtype": "int", "pkv_status": "int", "int32_t": "int", "unsigned": "uint",
            "int64_t": "int64", "size_t": "size", "float": "float", "void": "void"}[t]


def _ctypes_kind(t):
    if t is None:
        return "void"
    if t is ctypes.c_char_p:
        return "char_p"
    if t is ctypes.c_void_p or (isinstance(t, type) and issubclass(t, ctypes._Pointer)):
        return "ptr"
    return {ctypes.c_int: "int", ctypes.c_int32: "int", ctypes.c_uint: "uint", ctypes.c_int64: "int64",
            ctypes.c_size_t: "size", ctypes.c_float: "float"}[t]


def header_prototypes():
    """name -> (return kind, [parameter kinds]) for every PKV_API declaration."""
    text = re.sub(r"/\*.*?\*/", " ", open(HEADER).read(), flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    protos = {}
    for m in re.finditer(r"PKV_API\s+([\w\s\*]+?)\b(pkv_\w+)\s*\(([^)]*)\)\s*;", text):
        params = [p.strip() for p in m.group(3).split(",") if p.strip() and p.strip() != "void"]
        # a parameter's type is the declaration without its name
        kinds = [_c_kind(re.sub(r"\b\w+\s*$", "", p) if not p.rstrip().endswith("*") else p) for p in params]
        protos[m.group(2)] = (_c_kind(m.group(1)), kinds)
    return protos


def test_binding_signatures_match_the_header(lib):
    """Every ctypes declaration in the binding passes what the header's prototype takes:
    the same number of parameters, each a pointer, an int, a 64-bit int, a size or a float
    where the header says so, and the same return type."""
    protos = header_prototypes()
    assert sorted(protos) == declared_symbols()
    for name, (ret, params) in protos.items():
        fn = getattr(lib, name)
        got = [_ctypes_kind(t) for t in (fn.argtypes or [])]
        assert got == params, f"{name}: binding passes {got}, header declares {params}"
        assert _ctypes_kind(fn.restype) == ret, f"{name}: binding returns {fn.restype}, header {ret}"


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s(pkv_\w+)$", out, re.M))
    for name in declared_symbols():
        assert name in exported, name
        assert hasattr(lib, name)
    # nothing else leaks out of the library
    assert exported == set(declared_symbols())


def test_version_and_empty_error(lib):
    assert lib.pkv_version() == 100


def test_validation_rejects_before_launch(lib):
    null = ctypes.c_void_p(0)
    # unsupported head_dim
    st = lib.pkv_paged_attention_decode(null, null, null, null, null, 4, null, 2, 10, 8, 2, 96, 16, 10, 1.0, 0,
                                        null, 0, 0, null)
    assert st == pkv.PKV_ERR_UNSUPPORTED and b"head_dim" in lib.pkv_last_error()
    # heads not a multiple of KV heads
    st = lib.pkv_paged_attention_decode(null, null, null, null, null, 4, null, 2, 10, 7, 2, 128, 16, 10, 1.0, 0,
                                        null, 0, 0, null)
    assert st == pkv.PKV_ERR_INVALID
    # block size not built
    st = lib.pkv_paged_attention_decode(null, null, null, null, null, 4, null, 2, 10, 8, 2, 128, 12, 10, 1.0, 0,
                                        null, 0, 0, null)
    assert st == pkv.PKV_ERR_UNSUPPORTED
    # max_seq_len beyond the table width
    st = lib.pkv_paged_attention_decode(null, null, null, null, null, 4, null, 2, 65, 8, 2, 128, 16, 10, 1.0, 0,
                                        null, 0, 0, null)
    assert st == pkv.PKV_ERR_INVALID
    # partition size not a multiple of 64
    st = lib.pkv_paged_attention_decode(null, null, null, null, null, 4, null, 2, 10, 8, 2, 128, 16, 10, 1.0, 0,
                                        null, 0, 100, null)
    assert st == pkv.PKV_ERR_INVALID
    # null pointers
    st = lib.pkv_paged_attention_decode(null, null, null, null, null, 4, null, 2, 10, 8, 2, 128, 16, 10, 1.0, 0,
                                        null, 0, 64, null)
    assert st == pkv.PKV_ERR_INVALID and b"null" in lib.pkv_last_error()
    assert lib.pkv_paged_kv_append(null, null, null, null, null, -1, 4, 16, 2, 64, 0, null) == pkv.PKV_ERR_INVALID
    assert lib.pkv_paged_kv_append(null, null, null, null, null, 3, 4, 16, 2, 64, 0, null) == pkv.PKV_ERR_INVALID
    assert lib.pkv_paged_kv_append(null, null, null, null, null, 3, 4, 16, 2, 64, 7, null) == pkv.PKV_ERR_UNSUPPORTED
    assert lib.pkv_copy_blocks(None, None, -1, null, 1, 4, 16, 2, 64, 0, null) == pkv.PKV_ERR_INVALID
    # empty work is accepted without touching the device
    assert lib.pkv_paged_kv_append(null, null, null, null, null, 0, 4, 16, 2, 64, 0, null) == pkv.PKV_OK
    assert lib.pkv_copy_blocks(None, None, 0, null, 0, 4, 16, 2, 64, 0, null) == pkv.PKV_OK


def test_fused_and_verify_validation_rejects_before_launch(lib):
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(256)            # a non-null, aligned address that nothing dereferences

    def fused(head_dim=128, dt=0, kv_dt=0, k_scale=null, v_scale=null, sum_lens=0, ptr=fake, slots=fake, planned=1):
        # out, q, k, v, key_cache, value_cache, slot_mapping, tables, width, lens, B, max_len, sum, Hq, Hkv, d, bs,
        # num_blocks, scale, dt, kv_dt, k_scale, v_scale, workspace, workspace_bytes, partition, planned, stream
        return lib.pkv_paged_kv_append_decode(ptr, ptr, ptr, ptr, ptr, ptr, slots, fake, 4, fake, 2, 10, sum_lens, 8, 2,
                                              head_dim, 16, 10, 1.0, dt, kv_dt, k_scale, v_scale, null, 0, 0, planned,
                                              null)

    assert fused(sum_lens=-1) == pkv.PKV_ERR_INVALID
    # planned: 0, PKV_PLANNED (1) or PKV_PLANNED | PKV_INPUTS_READY (3); inputs-ready alone or other bits refused
    for bad in (pkv.INPUTS_READY, 4, 5, 7, -1):
        assert fused(planned=bad) == pkv.PKV_ERR_INVALID and b"planned" in lib.pkv_last_error()
    assert fused(kv_dt=1) == pkv.PKV_ERR_INVALID and b"kv_dt" in lib.pkv_last_error()   # 16-bit pools: kv_dt == dt
    assert fused(kv_dt=2) == pkv.PKV_ERR_INVALID                                          # E4M3 without scales
    assert fused(head_dim=96) == pkv.PKV_ERR_UNSUPPORTED
    assert fused(head_dim=64, kv_dt=2, k_scale=fake, v_scale=fake) == pkv.PKV_ERR_UNSUPPORTED   # E4M3: head_dim 128
    assert fused(ptr=null) == pkv.PKV_ERR_INVALID and b"null" in lib.pkv_last_error()
    assert fused(slots=null) == pkv.PKV_ERR_INVALID and b"null" in lib.pkv_last_error()
    assert fused(slots=ctypes.c_void_p(260)) == pkv.PKV_ERR_INVALID                      # slot_mapping 8-byte aligned
    # verify: a negative lengths' sum is refused
    st = lib.pkv_paged_attention_verify(fake, fake, fake, fake, fake, 4, fake, 2, 10, -1, 8, 2, 128, 16, 10, 1.0, 0, 4,
                                        null, 0, 0, null)
    assert st == pkv.PKV_ERR_INVALID

    def verify(nq=4, head_dim=128, ptr=fake):
        # out, q, key_cache, value_cache, tables, width, lens, B, max_len, sum, Hq, Hkv, d, bs, num_blocks, scale, dt,
        # num_queries, workspace, workspace_bytes, partition, stream
        return lib.pkv_paged_attention_verify(ptr, fake, fake, fake, fake, 4, fake, 2, 10, 0, 8, 2, head_dim, 16, 10,
                                              1.0, 0, nq, null, 0, 0, null)

    for nq in (0, -1, 65):                  # query tokens per sequence in [1, 64]
        assert verify(nq=nq) == pkv.PKV_ERR_INVALID and b"num_queries" in lib.pkv_last_error()
    assert verify(head_dim=96) == pkv.PKV_ERR_UNSUPPORTED
    assert verify(ptr=null) == pkv.PKV_ERR_INVALID

    def verify_fp8(k_scale=fake, v_scale=fake, head_dim=128, sum_lens=0):
        # as verify, with the scales before num_queries
        return lib.pkv_paged_attention_verify_fp8(fake, fake, fake, fake, fake, 4, fake, 2, 10, sum_lens, 8, 2,
                                                  head_dim, 16, 10, 1.0, 0, k_scale, v_scale, 4, null, 0, 0, null)

    assert verify_fp8(k_scale=null) == pkv.PKV_ERR_INVALID and b"k_scale" in lib.pkv_last_error()
    assert verify_fp8(v_scale=null) == pkv.PKV_ERR_INVALID
    assert verify_fp8(sum_lens=-5) == pkv.PKV_ERR_INVALID
    assert verify_fp8(head_dim=64) == pkv.PKV_ERR_UNSUPPORTED         # E4M3 pools: head_dim 128
    # a 128K-position batch at 64-position partitions (2048 per sequence, past the 512 the merge
    # holds) is refused before any driver call, naming the way out
    st = lib.pkv_paged_attention_decode(fake, fake, fake, fake, fake, 8192, fake, 2, 131072, 8, 2, 128, 16, 20000,
                                        1.0, 0, fake, 1 << 30, 64, null)
    assert st == pkv.PKV_ERR_UNSUPPORTED and b"use a larger partition_tokens" in lib.pkv_last_error()


def test_workspace_formula(lib):
    # explicit partition sizes need no device query
    B, Hq, Hkv, d = 16, 64, 8, 128
    pad = lambda x: (x + 255) // 256 * 256
    tickets = pad(4 * B * Hkv)                # one ticket per (sequence, KV head)
    # one partition: no partials, one 32-byte work-list entry per sequence
    assert lib.pkv_decode_workspace_bytes(B, Hq, Hkv, d, 512, 512) == tickets + pad(32 * B)
    n = lib.pkv_decode_workspace_bytes(B, Hq, Hkv, d, 4096, 512)
    sh = B * Hq * 8
    assert n == tickets + pad(32 * B * 8) + pad(sh * d * 4) + pad(sh * 8)
    # more than 8 query heads per KV head: one ticket per 8-head group
    assert lib.pkv_decode_workspace_bytes(2, 64, 2, d, 64, 64) == pad(4 * 2 * 2 * 4) + pad(32 * 2)
    # at most 4 query heads per KV head (shared-prefix units possible): one spare partition per row
    n = lib.pkv_decode_workspace_bytes(B, 32, Hkv, d, 4096, 512)
    sh = B * 32 * 9
    assert n == tickets + pad(32 * B * 9) + pad(sh * d * 4) + pad(sh * 8)
    assert lib.pkv_decode_workspace_bytes(B, Hq, Hkv, 96, 4096, 512) == ctypes.c_size_t(-1).value
    assert lib.pkv_decode_workspace_bytes(B, Hq, Hkv, d, 4096, 100) == ctypes.c_size_t(-1).value


def test_binding_refuses_cpu_tensors(lib):
    import torch
    t = torch.zeros(4, 16, 2, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        pkv.paged_kv_append(torch.zeros(1, 2, 64, dtype=torch.float16), torch.zeros(1, 2, 64, dtype=torch.float16),
                            t, t, torch.zeros(1, dtype=torch.int64))


def test_binding_refuses_tensors_on_two_devices(lib):
    """Every CUDA tensor of one call must sit on one device (the kernels run on
    that device and dereference every pointer there).  Stand-in tensors that
    report a CUDA device let this run without a GPU: the check raises before
    any pointer is read."""
    import torch

    class OnDevice(torch.Tensor):
        @property
        def is_cuda(self):
            return True

        @property
        def device(self):
            return self._dev

    def on(i, shape=(1,)):
        t = torch.Tensor._make_subclass(OnDevice, torch.zeros(shape))
        t._dev = torch.device("cuda", i)
        return t

    assert pkv._cuda_devices([on(0), [on(1), torch.zeros(1)], None, 3]) == {torch.device("cuda", 0),
                                                                               torch.device("cuda", 1)}
    assert pkv._cuda_devices([torch.zeros(1), [torch.zeros(1)]]) == set()
    with pytest.raises(ValueError, match="more than one device"):
        pkv.paged_kv_append(on(0), on(0), on(1), on(1), on(0))
    with pytest.raises(ValueError, match="more than one device"):
        pkv.copy_blocks([on(0)], [on(1)], on(0))
    with pytest.raises(ValueError, match="more than one device"):
        pkv.paged_attention_decode(on(0), on(0), on(0), on(0), on(0), on(1), max_seq_len=1)


def test_host_partition_rule_properties(lib):
    """The host's smallest partition size (pkv_decode_partition_tokens) over a grid
    of batch shapes, including 0 sequences, length 0 and lengths far past any
    configuration: always a multiple of 64 in [128, 4096], the range the decode
    call accepts, and the workspace for it is defined.  Without a GPU the rule
    takes 152 SMs and one resident CTA per SM."""
    for B in (0, 1, 4, 16, 64, 128, 768, 65535):
        for Hq, Hkv in ((4, 4), (32, 8), (64, 8), (8, 1)):
            for L in (0, 1, 50, 1024, 4096, 8192, 66000, 100000, 400000, 600000, 2 ** 21):
                for d in (64, 128):
                    p = lib.pkv_decode_partition_tokens(B, Hq, Hkv, d, L)
                    assert p % 64 == 0 and 128 <= p <= 4096, (B, Hq, Hkv, L, d, p)
                    assert lib.pkv_decode_workspace_bytes(B, Hq, Hkv, d, L, p) != ctypes.c_size_t(-1).value
                    # the automatic size never asks for more partitions than the call accepts (one
                    # sequence of 66000 positions over one KV head once got 128 positions: 516)
                    assert -(-L // p) <= 512, (B, Hq, Hkv, L, d, p)
    assert lib.pkv_decode_partition_tokens(4, 6, 4, 128, 100) < 0        # heads not a multiple of KV heads
    assert lib.pkv_decode_partition_tokens(4, 8, 2, 96, 100) < 0         # head_dim not built

