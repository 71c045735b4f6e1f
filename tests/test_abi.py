"""The C ABI: the library builds, loads, exports every symbol the header declares,
and rejects bad arguments on the host without touching a device.  CPU only."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dspark.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    import speculative_decoding_verification_dspark_gb300 as pkg
    return pkg.load()


def test_header_declares_the_five_calls():
    names = _declared()
    for n in ("dspark_schedule", "dspark_pack", "dspark_verify_attn", "dspark_accept",
              "dspark_compact"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    assert lib.dspark_status_string(0) == b"ok"
    assert lib.dspark_status_string(-1) == b"invalid argument"


def test_host_validation_without_device(lib):
    # NULL pointers and out-of-range sizes are rejected before any device work
    nul = None
    assert lib.dspark_schedule(nul, 1, nul, nul, 10, 4, 6, 32, 0, nul, nul, nul, nul, nul, nul) == -1
    assert lib.dspark_pack(nul, nul, nul, nul, nul, 0, 4, 6, 0, 8, nul, nul, nul, nul, nul, nul,
                           nul, nul) == -1
    # unsupported attention shape (head dim 96)
    assert lib.dspark_verify_attn(nul, nul, nul, nul, nul, 1, nul, 1, nul, nul, 1, 8, 8, 2, 96, 96,
                                  16, ctypes.c_float(0.1), 4, 9, nul, nul, nul, 0, nul) == -2
    # vocabulary not a multiple of 8
    fake = ctypes.c_void_p(4096)
    # pack + work list: NULL pointers; then valid pointers with an unsupported attention
    # shape (head dim 96); the planned attention validates as the standalone call
    assert lib.dspark_pack_plan(nul, nul, nul, nul, nul, 0, 4, 6, 0, 8, nul, nul, nul, nul, nul,
                                nul, nul, 8, 2, 128, 128, 8, 4, 7, nul, 0, nul) == -1
    assert lib.dspark_pack_plan(fake, fake, fake, fake, nul, 0, 4, 6, 0, 8, fake, fake, fake, nul,
                                fake, fake, fake, 8, 2, 96, 96, 8, 4, 7, fake, 1 << 20, nul) == -2
    assert lib.dspark_pack_plan(fake, fake, fake, fake, nul, 0, 4, 6, 0, 8, fake, fake, fake, nul,
                                fake, fake, fake, 8, 2, 128, 128, 8, 33, 7, fake, 1 << 20, nul) == -1
    assert lib.dspark_verify_attn_planned(nul, nul, nul, nul, nul, 1, nul, 1, nul, nul, 1, 8, 8, 2,
                                          96, 96, 16, ctypes.c_float(0.1), 4, 9, nul, nul, nul, 0,
                                          nul) == -2
    assert lib.dspark_accept(fake, fake, 0, 1001, fake, fake, fake, fake, fake, 0, 4, 6, 8, fake,
                             fake, fake, fake, nul, fake, 1 << 20, nul) == -2
    # the fixed-scratch variant: a problem larger than its scratch is refused (ENOSPACE)
    # on the host, and a small one passes validation up to the device check
    assert lib.dspark_accept_noalloc(fake, fake, 0, 151936, fake, fake, fake, fake, fake, 0, 4, 6,
                                     16384, fake, fake, fake, fake, nul, nul) == -4
    assert lib.dspark_accept_noalloc(fake, fake, 0, 1001, fake, fake, fake, fake, fake, 0, 4, 6, 8,
                                     fake, fake, fake, fake, nul, nul) == -2
    # block-accept estimate: NULL pointers, an unknown probability type, a mode out of range
    assert lib.dspark_block_accept_estimate(nul, fake, 0, 1024, fake, fake, fake, fake, fake, fake,
                                            0, 4, 6, 8, fake, fake, nul) == -1
    assert lib.dspark_block_accept_estimate(fake, fake, 7, 1024, fake, fake, fake, fake, fake, fake,
                                            0, 4, 6, 8, fake, fake, nul) == -1
    assert lib.dspark_block_accept_estimate(fake, fake, 0, 1024, fake, fake, fake, fake, fake, fake,
                                            3, 4, 6, 8, fake, fake, nul) == -1
    # Markov-head draft: NULL pointers, a rank other than 256, a vocabulary that is not a
    # multiple of 128, gamma above the maximum, misaligned logits
    ws = lib.dspark_markov_draft_workspace_size(1024)
    assert lib.dspark_markov_draft(nul, fake, fake, 256, fake, fake, 4, 6, 1024, fake, fake, fake,
                                   ws, nul) == -1
    assert lib.dspark_markov_draft(fake, fake, fake, 128, fake, fake, 4, 6, 1024, fake, fake, fake,
                                   ws, nul) == -2
    assert lib.dspark_markov_draft(fake, fake, fake, 256, fake, fake, 4, 6, 1000, fake, fake, fake,
                                   ws, nul) == -2
    assert lib.dspark_markov_draft(fake, fake, fake, 256, fake, fake, 4, 33, 1024, fake, fake, fake,
                                   ws, nul) == -1
    assert lib.dspark_markov_draft(ctypes.c_void_p(4100), fake, fake, 256, fake, fake, 4, 6, 1024,
                                   fake, fake, fake, ws, nul) == -1


def test_workspace_sizes_are_host_computable(lib):
    s = lib.dspark_verify_attn_workspace_size(32, 512, 32, 8, 128, 128, 8, 9)
    assert s > 0
    assert lib.dspark_verify_attn_workspace_size(64, 1024, 128, 1, 576, 512, 8, 9) > 0
    assert lib.dspark_verify_attn_workspace_size(32, 512, 32, 8, 96, 96, 8, 9) == 0
    assert lib.dspark_accept_workspace_size(32, 8, 512, 151936) > 0
    assert lib.dspark_compact_workspace_size(32) > 0
    assert lib.dspark_markov_draft_workspace_size(151936) > 0
    assert lib.dspark_markov_draft_workspace_size(151936) == lib.dspark_markov_draft_workspace_size(1024)
    assert lib.dspark_markov_draft_workspace_size(1000) == 0


def test_attention_workspace_follows_the_query_tile(lib):
    """A smaller block-rows hint (a smaller query tile, more row tiles per request)
    needs at least as many work items, so at least as large a workspace; a hint <= 0
    counts as one row, and the latent-KV shape ignores the hint."""
    ws = lambda h: lib.dspark_verify_attn_workspace_size(32, 512, 32, 8, 128, 128, 8, h)
    sizes = [ws(h) for h in (17, 9, 8, 4, 1)]
    assert all(a <= b for a, b in zip(sizes, sizes[1:])) and sizes[0] < sizes[-1]
    assert ws(0) == ws(-3) == ws(1)
    mla = lambda h: lib.dspark_verify_attn_workspace_size(64, 1024, 128, 1, 576, 512, 8, h)
    assert mla(9) == mla(1) == mla(0) > 0


def test_step_graph_rejects_bad_descriptors_on_the_host(lib):
    """The step graph's descriptor is checked before any CUDA work: NULL arguments,
    tiers that are not ascending or exceed the row capacity."""
    import speculative_decoding_verification_dspark_gb300 as pkg
    out = ctypes.c_void_p()
    assert lib.dspark_step_graph_create(None, ctypes.byref(out)) == -1
    d = pkg.StepDesc()
    d.B, d.gamma, d.max_rows = 4, 6, 32
    tiers = (ctypes.c_int32 * 3)(8, 16, 64)      # 64 > max_rows
    d.n_tiers, d.tiers_host, d.tiers = 3, ctypes.cast(tiers, ctypes.c_void_p), 4096
    assert lib.dspark_step_graph_create(ctypes.byref(d), ctypes.byref(out)) == -1
    tiers2 = (ctypes.c_int32 * 3)(8, 8, 16)      # not strictly ascending
    d.tiers_host = ctypes.cast(tiers2, ctypes.c_void_p)
    assert lib.dspark_step_graph_create(ctypes.byref(d), ctypes.byref(out)) == -1
    d.B = 0
    assert lib.dspark_step_graph_create(ctypes.byref(d), ctypes.byref(out)) == -1
    assert out.value is None
    assert lib.dspark_step_graph_destroy(None) == 0


def test_step_desc_layout_matches_the_header():
    """The binding's descriptor has the header's field order and size (every field of
    the C struct, in order, with the C alignment)."""
    import re
    import speculative_decoding_verification_dspark_gb300 as pkg
    text = open(HEADER).read()
    body = text[text.index("typedef struct dspark_step_desc {"):text.index("} dspark_step_desc;")]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = []
    for decl in body.split(";")[:-1]:
        decl = decl.split("{")[-1].strip()
        if not decl:
            continue
        head, *rest = [x.strip() for x in decl.split(",")]
        names.append(re.split(r"[\s*]+", head)[-1])
        names.extend(rest)
    assert [f[0] for f in pkg.StepDesc._fields_] == names
