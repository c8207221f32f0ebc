"""The TMA decode's shared-memory layout for every instance it launches, checked
on the host (nvcc, no GPU): the stage rings of the four sections, the header
(queries, block ids, loop state, barriers) and the code table never overlap;
the table starts at a 64 KB-aligned shared address, so that a code byte in
bits 8-15 of a byte permute with a per-lane register forms an entry's whole
address, and holds every entry the codes can index; everything fits the
227 KB a block may use; tiles sit on their swizzle and TMA alignments."""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "quantized_paged_kv_reshape_gb300", "csrc")

# (K side, V side, head_dim) of every launch_tma_inst in csrc/kvq_decode_tma_k_*.cu
INSTANCES = [
    ("S_BF16", "S_BF16", 64), ("S_BF16", "S_BF16", 128), ("S_BF16", "S_T2", 64),
    ("S_BF16", "S_T2", 128), ("S_BF16", "S_T3", 128), ("S_BF16", "S_T4", 64),
    ("S_BF16", "S_T4", 128), ("S_FP8", "S_FP8", 64), ("S_FP8", "S_FP8", 128),
    ("S_FP8", "S_T2", 64), ("S_FP8", "S_T2", 128), ("S_FP8", "S_T3", 128),
    ("S_FP8", "S_T4", 64), ("S_FP8", "S_T4", 128), ("S_NVFP4", "S_NVFP4", 64),
    ("S_NVFP4", "S_NVFP4", 128), ("S_T4", "S_T3", 128), ("S_T4", "S_T4", 64),
    ("S_T4", "S_T4", 128),
]
FIELDS = ("NW NST CPS SMEM LIMIT HEAD LUT LUT_OFF LUT_END LUT_ADDR LUT_ENTRIES R_KD R_VD R_KS R_VS "
          "OFF_MERGE MERGE_BYTES KTILE VTILE KSTILE VSTILE KCB VCB").split()


def test_instances_match_the_sources():
    found = set()
    for name in os.listdir(CSRC):
        if name.startswith("kvq_decode_tma_k_") and name.endswith(".cu"):
            with open(os.path.join(CSRC, name)) as f:
                found |= {(k, v, int(h)) for k, v, h in
                          re.findall(r"launch_tma_inst<(S_\w+), (S_\w+), (\d+)>", f.read())}
    assert found == set(INSTANCES)


@pytest.fixture(scope="module")
def layouts(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    d = tmp_path_factory.mktemp("tma_layout")
    body = []
    for k, v, hd in INSTANCES:
        for pk in ("true", "false"):
            body.append(f'  show<{k}, {v}, {hd}, {pk}>("{k} {v} {hd} {pk}");')
    src = d / "layout.cu"
    src.write_text(
        '#include "kvq_decode_tma.cuh"\n#include <cstdio>\nusing namespace kvq;\n'
        "template <int KS, int VS, int HD, bool PK> void show(const char* n) {\n"
        "  using C = TmCfg<KS, VS, HD, PK>;\n"
        '  std::printf("%s|%d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d\\n", n,\n'
        "    C::NW, C::NST, C::CPS, C::SMEM, C::LIMIT, C::HEAD, (int)C::LUT, C::LUT_OFF, C::LUT_END,\n"
        "    C::LUT_ADDR, C::LUT_ENTRIES, C::R_KD, C::R_VD, C::R_KS, C::R_VS, C::OFF_MERGE,\n"
        "    C::MERGE_BYTES, C::K::TILE, C::V::TILE, C::K::STILE, C::V::STILE, (int)C::K::CB,\n"
        "    (int)C::V::CB);\n}\nint main() {\n" + "\n".join(body) + "\n  return 0;\n}\n")
    exe = d / "layout"
    subprocess.run([nvcc, "-std=c++17", "--expt-relaxed-constexpr", "-I", CSRC,
                    "-I", os.path.join(ROOT, "include"), "-gencode",
                    "arch=compute_103a,code=sm_103a", str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    res = {}
    for line in out.splitlines():
        name, vals = line.split("|")
        res[name] = dict(zip(FIELDS, map(int, vals.split())))
    assert len(res) == 2 * len(INSTANCES)
    return res


def _overlap(a, b):
    return a[0] < b[1] and b[0] < a[1]


def test_regions_are_disjoint_and_fit(layouts):
    for name, c in layouts.items():
        n = c["NW"] * c["NST"]
        rings = {"kd": (c["R_KD"], c["R_KD"] + n * c["KTILE"]),
                 "vd": (c["R_VD"], c["R_VD"] + n * c["VTILE"]),
                 "ks": (c["R_KS"], c["R_KS"] + n * c["KSTILE"]),
                 "vs": (c["R_VS"], c["R_VS"] + n * c["VSTILE"])}
        rings = {k: r for k, r in rings.items() if r[1] > r[0]}
        head = (0, c["HEAD"])
        lut = (c["LUT_OFF"], c["LUT_END"]) if c["LUT"] else None
        keys = list(rings)
        for i, a in enumerate(keys):
            assert not _overlap(rings[a], head), (name, a)
            if lut:
                assert not _overlap(rings[a], lut), (name, a)
            assert rings[a][1] <= c["SMEM"], (name, a)
            for b in keys[i + 1:]:
                assert not _overlap(rings[a], rings[b]), (name, a, b)
        merge = (c["OFF_MERGE"], c["OFF_MERGE"] + c["MERGE_BYTES"])
        assert not _overlap(merge, head) and merge[1] <= c["SMEM"], name
        if lut:
            assert not _overlap(merge, lut), name
        assert c["SMEM"] <= c["LIMIT"] <= 227 * 1024, name
        assert c["NST"] >= 2 and c["NW"] in (4, 8, 12, 16), name


def test_code_table_placement(layouts):
    for name, c in layouts.items():
        if not c["LUT"]:
            continue
        assert c["LUT_ADDR"] % 0x10000 == 0, name           # index byte in bits 8-15, ORed in
        assert c["LUT_ADDR"] == 0x400 + c["LUT_OFF"], name   # dynamic shared memory starts at 0x400
        assert c["LUT_END"] - c["LUT_OFF"] == c["LUT_ENTRIES"] * 256, name
        ks, vs = name.split()[:2]
        # codes index up to 256 entries (4-bit pairs, 2-bit quads); the
        # 64-entry table serves Turbo3 pairs only, when it is the only table
        if c["LUT_ENTRIES"] == 64:
            assert vs == "S_T3" and not c["KCB"], name
        else:
            assert c["LUT_ENTRIES"] == 256, name


def test_tile_alignment(layouts):
    for name, c in layouts.items():
        assert c["R_KD"] % 1024 == 0 and c["R_VD"] % 1024 == 0, name   # swizzle atoms
        assert c["R_KS"] % 128 == 0 and c["R_VS"] % 128 == 0, name
        assert c["HEAD"] % 1024 == 0, name
