"""CPU-only checks of the C ABI: the library loads, exports every declared
symbol, and rejects bad arguments on the host before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ffa.h")


@pytest.fixture(scope="module")
def lib():
    from flexible_mask_flashattention_gb300 import build
    build.build()
    import flexible_mask_flashattention_gb300 as ffa
    return ffa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(ffa_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("ffa_plan_create", "ffa_plan_destroy", "ffa_plan_info", "ffa_plan_copy_csr", "ffa_fwd", "ffa_bwd",
                 "ffa_bwd_workspace_size", "ffa_status_string", "ffa_plan_check_status",
                 "ffa_plan_copy_bwd_items"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def declared_prototypes():
    """{name: (return type, [parameter types])} of every function in the header, each type reduced to
    a kind: ptr, i32, i64, u64, f32, f64."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    protos = {}
    for ret, name, params in re.findall(r"^\s*((?:const\s+)?[a-z_0-9]+\s*\*?)\s*(ffa_[a-z_0-9]+)\s*\(([^)]*)\)\s*;",
                                        text, flags=re.M):
        kinds = []
        for prm in (x.strip() for x in params.split(",") if x.strip() and x.strip() != "void"):
            typ = prm.rsplit(None, 1)[0] if "*" not in prm.rsplit(None, 1)[-1] else prm
            if "*" in prm or typ.endswith("ffa_plan_t"):
                kinds.append("ptr")
            else:
                kinds.append({"int32_t": "i32", "int64_t": "i64", "size_t": "u64", "float": "f32", "double": "f64",
                              "int": "i32", "ffa_status": "i32"}[typ.replace("const ", "").strip()])
        protos[name] = (re.sub(r"\s+", "", ret), kinds)
    return protos


def ctypes_kind(t):
    if t in (ctypes.c_void_p, ctypes.c_char_p) or (isinstance(t, type) and issubclass(t, ctypes._Pointer)):
        return "ptr"
    for kind, cls in (("i32", ctypes.c_int32), ("i64", ctypes.c_int64), ("u64", ctypes.c_uint64),
                      ("f32", ctypes.c_float), ("f64", ctypes.c_double)):
        if ctypes.sizeof(t) == ctypes.sizeof(cls) and t._type_ == cls._type_:
            return kind
    raise AssertionError(f"unmapped ctypes type {t}")


def test_binding_signatures_match_the_header(lib):
    """Every function the header declares is bound in _lib.py with the header's parameter kinds and
    return type (the binding's argtypes against the prototypes, parameter by parameter)."""
    protos = declared_prototypes()
    assert set(protos) == set(declared_functions())
    for name, (ret, kinds) in protos.items():
        f = getattr(lib, name)
        assert f.argtypes is not None, f"{name} is not declared in the binding"
        assert [ctypes_kind(t) for t in f.argtypes] == kinds, name
        want_ret = {"ffa_status": ctypes.c_int, "size_t": ctypes.c_size_t, "constchar*": ctypes.c_char_p}[ret]
        assert f.restype == want_ret, name


def test_boundary_calls_and_types_of_the_scope_table():
    """The boundary's calls and types: the plan / forward / backward calls with the tile-size struct,
    the status and mask-type enums with their values."""
    protos = declared_prototypes()
    assert protos["ffa_plan_create"][1] == ["ptr", "i64", "i64", "i64", "ptr", "ptr", "ptr"]
    assert protos["ffa_fwd"][1] == ["ptr", "ptr", "ptr", "i64", "i64", "i32", "i32", "i32", "ptr", "f32", "ptr",
                                    "ptr", "ptr"]
    assert protos["ffa_bwd"][1] == ["ptr"] * 6 + ["i64", "i64", "i32", "i32", "i32", "ptr", "f32"] + ["ptr"] * 4 + \
        ["u64", "ptr"]
    text = open(HEADER).read()
    assert re.search(r"typedef struct \{\s*int32_t fwd_bm, fwd_bn, bwd_bm, bwd_bn;\s*\} ffa_tile_cfg;", text)
    for name, val in (("FFA_OK", 0), ("FFA_ERR_INVALID_ARG", 1), ("FFA_ERR_INVALID_SLICE", 2),
                      ("FFA_ERR_OVERLAPPING_COVERAGE", 3), ("FFA_ERR_UNSUPPORTED", 4), ("FFA_ERR_OVERFLOW", 5),
                      ("FFA_ERR_CUDA", 6), ("FFA_ERR_DEVICE_CHECK", 7), ("FFA_MASK_FULL", 0),
                      ("FFA_MASK_CAUSAL", 1), ("FFA_MASK_INV_CAUSAL", 2), ("FFA_MASK_BI_CAUSAL", 3)):
        assert re.search(rf"\b{name} = {val}\b", text), name


def test_status_strings(lib):
    for code in range(8):
        assert lib.ffa_status_string(code)
    assert lib.ffa_status_string(3).decode().startswith("a (query, key) pair")


def _create(lib, slices, sq, sk, bm=128, bn=128, bbm=128, bbn=128):
    from flexible_mask_flashattention_gb300._lib import AttnSliceC, TileCfgC
    arr = (AttnSliceC * max(1, len(slices)))()
    for i, (a, b, c, d, t) in enumerate(slices):
        arr[i] = AttnSliceC(a, b, c, d, t, 0)
    h = ctypes.c_void_p()
    tiles = TileCfgC(bm, bn, bbm, bbn)
    code = lib.ffa_plan_create(arr, len(slices), sq, sk, ctypes.byref(tiles), None, ctypes.byref(h))
    return code, h


def test_host_validation_rejects_bad_slices(lib):
    assert _create(lib, [(0, 10, 0, 10, 4)], 10, 10)[0] == 2           # unknown mask type
    assert _create(lib, [(0, 11, 0, 10, 0)], 10, 10)[0] == 2           # q range past seqlen_q
    assert _create(lib, [(5, 4, 0, 10, 0)], 10, 10)[0] == 2            # start > end
    assert _create(lib, [(-1, 4, 0, 10, 0)], 10, 10)[0] == 2           # negative start
    assert _create(lib, [(0, 4, 0, 12, 0)], 10, 10)[0] == 2            # k range past seqlen_k
    assert _create(lib, [(0, 4, 0, 4, 0)], 10, 10, bm=96)[0] == 4      # tile not a power of two
    assert _create(lib, [(0, 4, 0, 4, 0)], 10, 10, bn=4)[0] == 4       # tile too small
    assert _create(lib, [(0, 4, 0, 4, 0)], 10, 10, bbm=2048)[0] == 4   # backward tile too large
    assert _create(lib, [(0, 4, 0, 4, 0)], 10, 10, bbn=24)[0] == 4     # backward tile not a power of two
    assert _create(lib, [], -1, 10)[0] == 1
    assert _create(lib, [], (1 << 30) + 1, 10)[0] == 5


def test_host_validation_rejects_double_coverage(lib):
    # two FULL slices sharing pair (2, 3)
    assert _create(lib, [(0, 4, 0, 4, 0), (2, 3, 3, 5, 0)], 4, 5)[0] == 3
    # a square CAUSAL slice keeps c <= r: FULL slices strictly right of the diagonal do not meet it ...
    assert _create(lib, [(0, 4, 0, 4, 1), (0, 1, 1, 4, 0), (1, 2, 2, 4, 0)], 4, 4)[0] != 3
    # ... but one touching the diagonal does
    assert _create(lib, [(0, 4, 0, 4, 1), (1, 2, 1, 4, 0)], 4, 4)[0] == 3
    # sink + window as in the sink-and-window workload; a window reaching one key into the sink overlaps
    assert _create(lib, [(0, 64, 0, 8, 0), (8, 24, 8, 24, 1), (24, 64, 9, 64, 3)], 64, 64)[0] != 3
    assert _create(lib, [(0, 64, 0, 8, 0), (8, 24, 8, 24, 1), (24, 64, 7, 64, 3)], 64, 64)[0] == 3


def test_double_coverage_detection_matches_oracle(lib):
    import oracle
    import workloads
    counts = {True: 0, False: 0}
    for seed in range(60):
        sq, sk = 20 + seed % 13, 25 + seed % 7
        sl = workloads.random_slices(seed, sq, sk, max_segments=3, max_pieces=3)
        extra = workloads.random_slices(seed + 999, sq, sk, max_segments=2, max_pieces=2)
        both = [s.as_tuple() for s in sl] + [s.as_tuple() for s in extra]
        code, h = _create(lib, both, sq, sk)
        if code == 0:
            lib.ffa_plan_destroy(h)
        disjoint = oracle.coverage_is_disjoint(both, sq, sk)
        counts[disjoint] += 1
        if disjoint:
            assert code != 3, (seed, both)   # valid input: proceeds to the GPU (fails here with FFA_ERR_CUDA)
        else:
            assert code == 3, (seed, both)
    assert counts[True] >= 5 and counts[False] >= 5, counts


def test_python_layer_fails_loudly_without_library(tmp_path):
    import flexible_mask_flashattention_gb300._lib as L
    with pytest.raises(L.FFAError):
        L.load_library(str(tmp_path / "missing.so"))


def test_bwd_workspace_size(lib):
    # the header's layout: fp32 dq [sq][hq][d], lse and D [hq][sq rounded up to 128], fp32 dk and dv
    # [sk][hkv][d], each part 256-byte aligned; 0 for negative or zero sizes
    def a256(x):
        return (x + 255) // 256 * 256
    for sq, sk, hq, hkv, d in [(4096, 4096, 16, 4, 128), (4096, 4096, 16, 4, 64), (1000, 777, 3, 1, 64),
                               (1, 1, 1, 1, 128), (0, 5, 2, 2, 128), (130, 0, 8, 8, 64)]:
        sq_pad = (sq + 127) // 128 * 128
        want = a256(sq * hq * d * 4) + 2 * a256(sq_pad * hq * 4) + 2 * a256(sk * hkv * d * 4)
        assert lib.ffa_bwd_workspace_size(sq, sk, hq, hkv, d) == want
    for bad in [(-1, 5, 2, 2, 128), (5, -1, 2, 2, 128), (5, 5, 0, 2, 128), (5, 5, 2, 0, 128), (5, 5, 2, 2, 0)]:
        assert lib.ffa_bwd_workspace_size(*bad) == 0
    # the allocation-free backward's documented example: 4096 tokens, Hq 16, Hkv 4, d 128 need 48.5 MiB,
    # inside its 64 MiB array
    assert lib.ffa_bwd_workspace_size(4096, 4096, 16, 4, 128) == int(48.5 * 2 ** 20) < 64 * 2 ** 20
