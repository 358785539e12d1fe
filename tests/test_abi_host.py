"""Host-side tests of the C ABI (no GPU): the library loads, exports every symbol
declared in include/dplr.h, validates descriptors and rejects bad arguments before
launching anything."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dplr.h")


@pytest.fixture(scope="module")
def sdl():
    from structured_decay_linear_gb300 import build as nvbuild
    nvbuild.build()
    import structured_decay_linear_gb300 as s
    s.library()
    return s


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"DPLR_API\s+[\w\s\*]*?\b(dplr_\w+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    syms = declared_symbols()
    for name in ("dplr_la_forward", "dplr_la_workspace_size", "dplr_status_string", "dplr_la_chunk_maps",
                 "dplr_la_state_scan", "dplr_la_check", "dplr_la_kernel_count", "dplr_la_stage_workspace_size"):
        assert name in syms


def test_library_exports_every_declared_symbol(sdl):
    lib = sdl.library()
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} declared in dplr.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", sdl.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (dplr_\w+)", out))
    assert set(declared_symbols()) == exported, f"exported {sorted(exported)} vs declared {declared_symbols()}"


def test_header_compiles_as_c():
    src = '#include "dplr.h"\nint main(void){ dplr_desc d; (void)d; return (int)sizeof(dplr_desc) - 40; }\n'
    path = "/tmp/_dplr_hdr_test.c"
    with open(path, "w") as f:
        f.write(src)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), path, "-o",
                    "/tmp/_dplr_hdr_test"], check=True)
    assert subprocess.run(["/tmp/_dplr_hdr_test"]).returncode == 0


def test_path_names(sdl):
    assert sdl.dplr_la_path(sdl.make_desc("gdn", "bf16", 8, 16, 8192, 128, 128)) == "gdn_fused_tcgen05"
    assert sdl.dplr_la_path(sdl.make_desc("hdla", "bf16", 1, 16, 131072, 128, 128)) == "hdla_tcgen05"
    assert sdl.dplr_la_path(sdl.make_desc("hdla", "bf16", 1, 1, 64, 64, 64)) == "two_stage_fp32"
    assert sdl.dplr_la_path(sdl.make_desc("generic", "f32", 2, 8, 8192, 64, 64, 4, 2)) == "generic_tcgen05"
    assert sdl.dplr_la_path(sdl.make_desc("generic", "f32", 1, 1, 64, 64, 64, 8, 2)) == "two_stage_fp32"
    assert sdl.dplr_la_path(sdl.make_desc("generic", "f32", 1, 1, 64, 32, 32, 4, 2)) == "two_stage_fp32"
    assert sdl.dplr_la_path(sdl.make_desc("gdn", "f32", 1, 1, 8, 48, 32)) == ""


def test_status_strings(sdl):
    for code in range(6):
        assert sdl.status_string(code).startswith("DPLR_")
    assert "unknown" in sdl.status_string(99)


@pytest.mark.parametrize("mode,dt,B,H,T,dk,dv,r,p,expect", [
    ("gdn", "f32", 1, 2, 256, 32, 32, 1, 1, 0),
    ("hdla", "bf16", 4, 16, 4096, 128, 128, 2, 1, 0),
    ("generic", "f32", 2, 8, 8192, 64, 64, 4, 2, 0),
    ("generic", "bf16", 1, 1, 10, 128, 64, 8, 8, 0),
    ("generic", "f32", 1, 1, 0, 32, 32, 1, 0, 0),
    ("gdn", "f32", 1, 1, 8, 48, 32, 1, 1, 2),       # dk not in {32, 64, 128}
    ("gdn", "f32", 1, 1, 8, 32, 256, 1, 1, 2),      # dv too large
    ("gdn", "f32", 1, 1, 8, 32, 32, 2, 1, 1),       # GDN rank is fixed
    ("hdla", "f32", 1, 1, 8, 32, 32, 1, 1, 1),      # HDLA rank is fixed
    ("generic", "f32", 1, 1, 8, 32, 32, 9, 1, 2),   # rank above 8
    ("generic", "f32", 1, 1, 8, 32, 32, 0, 1, 2),   # generic needs r_ab >= 1
    ("gdn", "f32", 0, 1, 8, 32, 32, 1, 1, 1),       # empty batch
    ("gdn", "f32", 1, 1, -1, 32, 32, 1, 1, 1),      # negative length
    # the largest shared-memory footprints of the two-stage kernels must still be accepted
    ("gdn", "f32", 1, 1, 64, 128, 128, 1, 1, 0),    # 64-token WY blocks with d = 128
    ("generic", "f32", 1, 1, 64, 128, 128, 4, 2, 0),
    ("generic", "f32", 1, 1, 64, 128, 128, 8, 8, 0),
])
def test_descriptor_validation(sdl, mode, dt, B, H, T, dk, dv, r, p, expect):
    d = sdl.make_desc(mode, dt, B, H, T, dk, dv, r, p)
    assert sdl.dplr_la_check(d) == expect
    ws = sdl.dplr_la_workspace_size(d)
    if expect != 0:
        assert ws == 0
    elif T > 0:
        assert ws > 0


def test_bad_enum_and_chunk(sdl):
    d = sdl.make_desc("gdn", "f32", 1, 1, 8, 32, 32)
    d.mode = 7
    assert sdl.dplr_la_check(d) == sdl.dplr.DPLR_ERR_INVALID_ARG
    d = sdl.make_desc("gdn", "f32", 1, 1, 8, 32, 32)
    d.in_dtype = 5
    assert sdl.dplr_la_check(d) == sdl.dplr.DPLR_ERR_INVALID_ARG
    d = sdl.make_desc("gdn", "f32", 1, 1, 8, 32, 32, chunk=32)
    assert sdl.dplr_la_check(d) == sdl.dplr.DPLR_ERR_UNSUPPORTED
    assert sdl.library().dplr_la_check(None) == sdl.dplr.DPLR_ERR_INVALID_ARG


def test_workspace_grows_with_length(sdl):
    sizes = [sdl.dplr_la_stage_workspace_size(sdl.make_desc("hdla", "bf16", 1, 2, T, 128, 128)) for T in (64, 128, 4096)]
    assert sizes[0] < sizes[1] < sizes[2]
    assert all(s % 256 == 0 for s in sizes)


FAKE = 1 << 20   # 16-byte aligned, never dereferenced: validation fails before any launch


def _fwd(sdl, d, **kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, decay=FAKE, beta=FAKE, A=None, Bm=None, K=None, V=None, S0=None,
                o=FAKE, S_T=None, workspace=FAKE, ws_bytes=sdl.dplr_la_workspace_size(d), stream=None)
    args.update(kw)
    return sdl.dplr_la_forward(d, **args)


@pytest.mark.parametrize("field", ["q", "k", "v", "decay", "beta", "o"])
def test_forward_rejects_null_input_before_launch(sdl, field):
    d = sdl.make_desc("hdla", "bf16", 1, 1, 64, 32, 32)
    assert _fwd(sdl, d, **{field: None}) == sdl.dplr.DPLR_ERR_INVALID_ARG


@pytest.mark.parametrize("field", ["q", "k", "decay", "o", "S0", "S_T"])
def test_forward_rejects_misaligned_pointer(sdl, field):
    d = sdl.make_desc("hdla", "bf16", 1, 1, 64, 32, 32)
    assert _fwd(sdl, d, **{field: FAKE + 4}) == sdl.dplr.DPLR_ERR_INVALID_ARG


def test_forward_rejects_small_or_missing_workspace(sdl):
    d = sdl.make_desc("gdn", "f32", 1, 1, 64, 32, 32)
    need = sdl.dplr_la_workspace_size(d)
    assert _fwd(sdl, d, ws_bytes=need - 1) == sdl.dplr.DPLR_ERR_WORKSPACE
    assert _fwd(sdl, d, workspace=None) == sdl.dplr.DPLR_ERR_WORKSPACE
    assert _fwd(sdl, d, workspace=FAKE + 16) == sdl.dplr.DPLR_ERR_WORKSPACE


def test_generic_requires_factor_pointers(sdl):
    d = sdl.make_desc("generic", "f32", 1, 1, 64, 32, 32, 2, 1)
    base = dict(k=None, v=None, beta=None, A=FAKE, Bm=FAKE, K=FAKE, V=FAKE)
    for field in ("A", "Bm", "K", "V"):
        kw = dict(base)
        kw[field] = None
        assert _fwd(sdl, d, **kw) == sdl.dplr.DPLR_ERR_INVALID_ARG
    d0 = sdl.make_desc("generic", "f32", 1, 1, 64, 32, 32, 2, 0)   # r_kv = 0: K, V unused
    kw = dict(base)
    kw.update(K=None, V=None, q=None)
    assert _fwd(sdl, d0, **kw) == sdl.dplr.DPLR_ERR_INVALID_ARG   # q still required


def test_stage_entry_points_validate(sdl):
    d = sdl.make_desc("gdn", "f32", 1, 1, 64, 32, 32)
    ws = sdl.dplr_la_workspace_size(d)
    assert sdl.dplr_la_chunk_maps(d, None, FAKE, FAKE, FAKE, FAKE, None, None, None, None, FAKE, FAKE, ws,
                                  None) == sdl.dplr.DPLR_ERR_INVALID_ARG
    ws = sdl.dplr_la_stage_workspace_size(d)
    assert sdl.dplr_la_state_scan(d, None, FAKE, None, FAKE, ws - 1, None) == sdl.dplr.DPLR_ERR_WORKSPACE
    assert sdl.dplr_la_state_scan(d, FAKE + 8, FAKE, None, FAKE, ws, None) == sdl.dplr.DPLR_ERR_INVALID_ARG


def test_fused_path_workspace_is_a_status_word(sdl):
    d = sdl.make_desc("gdn", "bf16", 8, 16, 8192, 128, 128)
    assert sdl.dplr_la_workspace_size(d) == 256
    assert sdl.dplr_la_stage_workspace_size(d) > 256
    assert sdl.dplr_la_kernel_count(d) == 1
    assert _fwd(sdl, d, ws_bytes=255) == sdl.dplr.DPLR_ERR_WORKSPACE


def test_kernel_count(sdl):
    assert sdl.dplr_la_kernel_count(sdl.make_desc("gdn", "f32", 1, 1, 64, 32, 32)) >= 1
    assert sdl.dplr_la_kernel_count(sdl.make_desc("gdn", "f32", 1, 1, 64, 48, 32)) == 0


def test_host_workspace_size_validates_groups_and_slots(sdl):
    d = sdl.make_desc("gdn", "bf16", 2, 8, 256, 128, 128)
    assert sdl.dplr_la_host_workspace_size(d, 4, 2) > 0
    assert sdl.dplr_la_host_workspace_size(d, 3, 2) == 0      # 16 heads are not a multiple of 3
    assert sdl.dplr_la_host_workspace_size(d, 0, 2) == 0
    assert sdl.dplr_la_host_workspace_size(d, 4, 0) == 0
    assert sdl.dplr_la_host_workspace_size(d, 4, 9) == 0
    # one slot per group at most: more slots than groups cost no more
    assert sdl.dplr_la_host_workspace_size(d, 2, 8) == sdl.dplr_la_host_workspace_size(d, 2, 2)
    # slots scale the size linearly
    assert sdl.dplr_la_host_workspace_size(d, 4, 2) == 2 * sdl.dplr_la_host_workspace_size(d, 4, 1)


def test_forward_host_rejects_bad_arguments_before_launch(sdl):
    d = sdl.make_desc("gdn", "bf16", 1, 4, 128, 128, 128)
    need = sdl.dplr_la_host_workspace_size(d, 2, 2)
    fake = 1 << 20      # never dereferenced: every check below comes first
    args = [fake] * 5 + [None] * 4 + [None, fake, None]
    call = lambda staging, nbytes, groups, slots, a=args: sdl.dplr_la_forward_host(d, *a, staging, nbytes, groups,
                                                                                    slots, None)
    assert call(fake, need, 3, 2) == sdl.dplr.DPLR_ERR_INVALID_ARG        # groups does not divide B*H
    assert call(fake, need, 2, 0) == sdl.dplr.DPLR_ERR_INVALID_ARG        # no slot
    assert call(fake, 4096, 2, 2) == sdl.dplr.DPLR_ERR_WORKSPACE          # staging too small
    assert call(fake + 16, need, 2, 2) == sdl.dplr.DPLR_ERR_WORKSPACE     # staging misaligned
    assert call(None, need, 2, 2) == sdl.dplr.DPLR_ERR_WORKSPACE
    no_k = [fake, None] + [fake] * 3 + [None] * 4 + [None, fake, None]
    assert call(fake, need, 2, 2, no_k) == sdl.dplr.DPLR_ERR_INVALID_ARG  # k missing


def test_host_seq_workspace_size(sdl):
    """Staging of the sequence-segmented host path: two state buffers plus one slot per segment in flight."""
    d = sdl.make_desc("gdn", "bf16", 2, 4, 1000, 128, 128)
    assert sdl.dplr_la_host_seq_workspace_size(d, 0, 2) == 0
    assert sdl.dplr_la_host_seq_workspace_size(d, 4, 0) == 0
    assert sdl.dplr_la_host_seq_workspace_size(d, 4, 9) == 0
    one, two = sdl.dplr_la_host_seq_workspace_size(d, 4, 1), sdl.dplr_la_host_seq_workspace_size(d, 4, 2)
    state = 2 * 4 * 128 * 128 * 4
    assert one > 2 * state and two - one == one - 2 * state          # slots add one slot each
    # 1000 tokens in 4 segments: 256-token segments, so 4 of them; slots beyond that cost nothing
    assert sdl.dplr_la_host_seq_workspace_size(d, 4, 8) == sdl.dplr_la_host_seq_workspace_size(d, 4, 4)
    # 3 segments of 1000 tokens round up to 384 tokens each: 3 segments
    assert sdl.dplr_la_host_seq_workspace_size(d, 3, 8) == sdl.dplr_la_host_seq_workspace_size(d, 3, 3)
    assert sdl.dplr_la_host_seq_workspace_size(sdl.make_desc("gdn", "bf16", 1, 2, 0, 128, 128), 4, 2) > 0


def test_host_path_default_segments(sdl):
    """Sequence segments of the segmented host path: 4 up to 32K tokens, then one per 8K tokens, at most 16."""
    ds = sdl.dplr.default_segments
    assert [ds(t) for t in (64, 4096, 8192, 16384, 32767)] == [4] * 5
    assert [ds(t) for t in (32768, 65536, 131072, 1 << 20)] == [4, 8, 16, 16]


def test_forward_host_seq_rejects_bad_arguments_before_launch(sdl):
    d = sdl.make_desc("gdn", "bf16", 1, 4, 128, 128, 128)
    need = sdl.dplr_la_host_seq_workspace_size(d, 2, 2)
    fake = 1 << 20      # never dereferenced: every check below comes first
    args = [fake] * 5 + [None] * 4 + [None, fake, None]
    call = lambda staging, nbytes, segments, slots, a=args: sdl.dplr_la_forward_host_seq(
        d, *a, staging, nbytes, segments, slots, None)
    assert call(fake, need, 0, 2) == sdl.dplr.DPLR_ERR_INVALID_ARG        # no segment
    assert call(fake, need, 2, 0) == sdl.dplr.DPLR_ERR_INVALID_ARG        # no slot
    assert call(fake, need, 2, 9) == sdl.dplr.DPLR_ERR_INVALID_ARG        # too many slots
    assert call(fake, 4096, 2, 2) == sdl.dplr.DPLR_ERR_WORKSPACE          # staging too small
    assert call(fake + 16, need, 2, 2) == sdl.dplr.DPLR_ERR_WORKSPACE     # staging misaligned
    assert call(None, need, 2, 2) == sdl.dplr.DPLR_ERR_WORKSPACE
    no_k = [fake, None] + [fake] * 3 + [None] * 4 + [None, fake, None]
    assert call(fake, need, 2, 2, no_k) == sdl.dplr.DPLR_ERR_INVALID_ARG  # k missing


def test_host_path_default_groups(sdl):
    """Head groups of the host-buffer path: at least 16 heads per group on the fused kernel, 32 on
    the two-stage kernels, and at most 16 groups."""
    dg = sdl.dplr.default_groups
    assert dg(sdl.make_desc("gdn", "bf16", 8, 16, 8192, 128, 128)) == 8
    assert dg(sdl.make_desc("hdla", "bf16", 4, 16, 4096, 128, 128)) == 2
    assert dg(sdl.make_desc("hdla", "bf16", 1, 16, 4096, 128, 128)) == 1
    assert dg(sdl.make_desc("gdn", "bf16", 32, 16, 1024, 128, 128)) == 16
