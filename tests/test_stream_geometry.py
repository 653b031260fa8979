"""Host checks of the decode stream's shared-memory geometry (csrc/stream_geom.h).

The header is plain constexpr C++ shared by the host and the kernel. A small
host program built on it with g++ lists, for every code width, group size and
padded token count, the ring (slots, slot bytes), the barrier, record and
partial-sum areas and the staged-activation room. The test checks that each
layout fits the thread block's shared memory, that the ring keeps the depth
and copy sizes the kernel relies on, and that the staging room holds the
activation buffers the chained launch plans for the 7B and 70B layer widths.
(A probe copy of the stream with 64 KiB slots once overflowed shared memory at
two or more tokens; the kernel now refuses such a layout at compile time, and
this test catches it before any CUDA build.)
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GEOM = os.path.join(ROOT, "weight_only_bit_04_b300", "csrc", "stream_geom.h")

PROGRAM = r"""
#define __host__
#define __device__
#include <cstdio>
#include <initializer_list>
#include GEOM_HEADER
using namespace w4a16;
int main() {
  std::printf("smem %d budget %d\n", kStreamSmem, kStreamRingBudget);
  for (int bits : {3, 4, 8})
    for (int gs : {32, 64, 128})
      for (int mp : {1, 2, 4, 8, 16})
        std::printf("%d %d %d %d %d %d %d %d %d %d\n", bits, gs, mp, stream_cu(bits, gs), stream_unit_code(bits, gs),
                    stream_slot_bytes(bits, gs), stream_slots(bits, gs), stream_part_off(bits, gs),
                    stream_x_off(bits, gs, mp), stream_x_bytes(bits, gs, mp));
  for (int K : {4096, 11008, 8192, 28672})
    for (int M : {1, 16})
      std::printf("xbuf %d %d %lld\n", K, M, stream_x_buf(K, M, 128));
  return 0;
}
"""


@pytest.fixture(scope="module")
def geometry(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("geom")
    src, exe = d / "geom.cpp", d / "geom"
    src.write_text(PROGRAM)
    subprocess.run([cxx, "-std=c++17", f'-DGEOM_HEADER="{GEOM}"', str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines()
    smem, budget = (int(v) for v in out[0].split()[1::2])
    rows, xbuf = [], {}
    for line in out[1:]:
        f = line.split()
        if f[0] == "xbuf":
            xbuf[(int(f[1]), int(f[2]))] = int(f[3])
        else:
            rows.append(dict(zip(("bits", "gs", "mp", "cu", "unit", "slot", "slots", "part_off", "x_off", "x_bytes"),
                                 (int(v) for v in f))))
    return smem, budget, rows, xbuf


def test_every_layout_fits_the_block(geometry):
    smem, _, rows, _ = geometry
    assert smem <= 227 * 1024
    assert len(rows) == 3 * 3 * 5
    for r in rows:
        assert r["slots"] * r["slot"] <= r["part_off"] <= r["x_off"] <= smem, r
        assert r["x_bytes"] == smem - r["x_off"] >= 0, r


def test_ring_depth_and_copy_sizes(geometry):
    _, budget, rows, _ = geometry
    for r in rows:
        cu = r["cu"]
        assert cu & (cu - 1) == 0 and 8 <= cu <= 32, r           # power-of-two boxes of at most 32 units
        assert cu % 8 == 0                                        # every consumer warp takes whole units
        assert r["slots"] >= 3, r                                 # copies in flight while one slot is computed
        assert r["slots"] * r["slot"] <= budget, r
        assert cu * r["unit"] <= 32 * 1024, r                     # a slot's codes within 32 KiB
        assert r["slot"] % 128 == 0 and r["part_off"] % 128 == 0  # aligned regions


def test_activation_room_holds_two_buffers_for_the_7b_and_70b_widths(geometry):
    """At one token the 7B widths (4096, 11008) and the 70B pair of 8192 and
    28672 fit two staged buffers side by side, so the next layer's activations
    land while the current one computes."""
    _, _, rows, xbuf = geometry
    room = next(r["x_bytes"] for r in rows if r["bits"] == 4 and r["gs"] == 128 and r["mp"] == 1)
    assert xbuf[(4096, 1)] + xbuf[(11008, 1)] <= room
    assert xbuf[(8192, 1)] + xbuf[(28672, 1)] <= room
    assert 2 * xbuf[(11008, 1)] <= room
