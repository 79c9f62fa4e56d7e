"""The C-ABI library builds, loads and exports every symbol include/sdverify.h
declares; host-side argument checks reject bad calls without a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from speculative_decoding_verify_gb300 import build as b
    b.build()
    import speculative_decoding_verify_gb300 as sdv
    return sdv.lib()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "sdverify.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sd_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_verify_calls():
    syms = declared_symbols()
    for name in ("sd_repack_weights", "sd_rmsnorm_quant_acts", "sd_qmatmul_multipos", "sd_head_logits",
                 "sd_accept_greedy", "sd_accept_sample"):
        assert name in syms


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), name


def test_binding_types_every_declared_call(L):
    """Each declared call has its argument types set in the binding (ctypes would otherwise pass
    floats and 64-bit integers wrongly)."""
    for name in declared_symbols():
        assert getattr(L, name).argtypes is not None, name


def test_status_strings_and_version(L):
    assert L.sd_abi_version() == 5
    assert L.sd_status_string(0) == b"ok"
    assert L.sd_status_string(4) == b"device wait timed out"


def test_repacked_sizes(L):
    # 4-bit: 576 B per (32-row tile, block); Q8_0: 1088 B; tails padded to whole tiles
    assert L.sd_repacked_bytes(1, 5120, 5120, 0) == 160 * 160 * 576
    assert L.sd_repacked_bytes(0, 151936, 5120, 0) == 4748 * 160 * 1088
    assert L.sd_repacked_bytes(1, 33, 64, 0) == 2 * 2 * 576
    assert L.sd_repacked_bytes(1, 2 * 17408, 5120, 1) == 544 * 2 * 160 * 576
    assert L.sd_repacked_bytes(1, 5120, 100, 0) == 0      # k_in % 32 != 0
    assert L.sd_repacked_bytes(1, 7, 64, 1) == 0          # odd n_out with the pair flag
    assert L.sd_repacked_bytes(7, 32, 64, 0) == 0         # unknown format


def test_argument_checks_reject_without_launching(L):
    p = ctypes.c_void_p(256)  # never dereferenced: validation fails first
    mis = ctypes.c_void_p(257)
    # qmatmul: M out of range, misaligned weights, k_in % 32, missing y for EPI_NONE
    assert L.sd_qmatmul_multipos(1, p, 64, 64, p, p, 17, p, None, 0, 0, None, None, p, 1 << 20, None) == 2
    assert L.sd_qmatmul_multipos(1, p, 64, 64, p, p, 0, p, None, 0, 0, None, None, p, 1 << 20, None) == 1
    assert L.sd_qmatmul_multipos(1, mis, 64, 64, p, p, 5, p, None, 0, 0, None, None, p, 1 << 20, None) == 1
    assert L.sd_qmatmul_multipos(1, p, 64, 48, p, p, 5, p, None, 0, 0, None, None, p, 1 << 20, None) == 1
    assert L.sd_qmatmul_multipos(1, p, 64, 64, p, p, 5, None, None, 0, 0, None, None, p, 1 << 20, None) == 1
    # requant epilogue: col0 not a multiple of 32
    assert L.sd_qmatmul_multipos(1, p, 64, 64, p, p, 5, None, None, 1, 16, p, p, p, 1 << 20, None) == 1
    # SiLU epilogue needs the 4-bit format and no residual
    assert L.sd_qmatmul_multipos(0, p, 64, 64, p, p, 5, None, None, 2, 0, p, p, p, 1 << 20, None) == 2
    assert L.sd_qmatmul_multipos(1, p, 64, 64, p, p, 5, None, p, 2, 0, p, p, p, 1 << 20, None) == 1
    # too-small workspace
    assert L.sd_qmatmul_multipos(1, p, 64, 64, p, p, 5, p, None, 0, 0, None, None, p, 0, None) == 1
    # head: non-positive temperature, M > 16
    assert L.sd_head_logits(p, 4096, 1024, p, p, 5, ctypes.c_float(0.0), p, p, p, p, p, 1 << 24, None) == 1
    assert L.sd_head_logits(p, 4096, 1024, p, p, 17, ctypes.c_float(1.0), p, p, p, p, p, 1 << 24, None) == 2
    # accept: K out of range, only one of the two statistics
    assert L.sd_accept_sample(p, 16, 16, None, None, None, p, ctypes.c_float(1.0), 0, 0, p, p, None) == 1
    assert L.sd_accept_sample(p, 16, 2, p, None, None, p, ctypes.c_float(1.0), 0, 0, p, p, None) == 1
    assert L.sd_accept_greedy(p, p, None, 17, p, p, None) == 1
    # rmsnorm: ldx < K
    assert L.sd_rmsnorm_quant_acts(p, 16, p, ctypes.c_float(1e-6), 5, 32, p, p, None) == 1
    assert L.sd_debug_wait_timeout(0, None) == 1
    # attention: S_max too small, unsupported D or M, misaligned q; commit without a count
    assert L.sd_kv_append(p, p, 5, 8, 128, p, p, 100, 96, None) == 1
    assert L.sd_attn_decode(p, p, p, 5, 8, 8, 96, 1000, 10, None, p, p, 1 << 20, None) == 2
    assert L.sd_attn_decode(p, p, p, 17, 8, 8, 128, 1000, 10, None, p, p, 1 << 20, None) == 2
    assert L.sd_attn_decode(p, p, p, 5, 12, 8, 128, 1000, 10, None, p, p, 1 << 20, None) == 1
    assert L.sd_attn_decode(mis, p, p, 5, 8, 8, 128, 1000, 10, None, p, p, 1 << 20, None) == 1
    assert L.sd_kv_commit(p, p, 8, 128, 1000, 10, 5, p, None, None) == 1
    assert L.sd_kv_commit(p, p, 8, 512, 1000, 10, 5, p, p, None) == 1
    # shortlist: misaligned head, hidden % 32, M out of range, missing argmax
    assert L.sd_shortlist_build(mis, 4096, 1024, p, p, p, None) == 1
    assert L.sd_shortlist_build(p, 4096, 1000, p, p, p, None) == 1
    assert L.sd_shortlist_build(p, 0, 1024, p, p, p, None) == 1
    assert L.sd_head_shortlist(p, p, p, p, 4096, 1024, p, p, 17, p, None, p, 1 << 24, None) == 2
    assert L.sd_head_shortlist(p, p, p, p, 4096, 1024, p, p, 0, p, None, p, 1 << 24, None) == 1
    assert L.sd_head_shortlist(p, p, p, mis, 4096, 1024, p, p, 5, p, None, p, 1 << 24, None) == 1
    assert L.sd_head_shortlist(p, p, p, p, 4096, 1024, p, p, 5, None, None, p, 1 << 24, None) == 1


def test_pass_structs_match_the_header(tmp_path):
    """The binding's ctypes mirrors of sd_layer, sd_pass_desc and sd_pass have the C layout: every
    field offset and the sizes, as gcc lays out the header."""
    import shutil
    import subprocess
    import speculative_decoding_verify_gb300 as sdv
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    structs = {"sd_layer": sdv.SdLayer, "sd_pass_desc": sdv.SdPassDesc, "sd_pass": sdv.SdPass}
    lines = ['#include <stdio.h>', '#include "sdverify.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for cname, py in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for f, _ in py._fields_:
            assert got[(cname, f)] == getattr(py, f).offset, (cname, f)
