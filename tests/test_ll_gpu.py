"""LL / LL128 kernels vs the oracle: wire bytes exactly, unpack-reduce exactly."""
import numpy as np
import pytest

import oracle
import collective_all_reduce_rank_gb300 as rra
from collective_all_reduce_rank_gb300 import inputs

pytestmark = pytest.mark.gpu

FMT = {
    "ll": (rra.rra_ll_pack, rra.rra_ll_unpack, rra.rra_ll_wire_bytes, oracle.ll_pack, oracle.ll_unpack),
    "ll128": (rra.rra_ll128_pack, rra.rra_ll128_unpack, rra.rra_ll128_wire_bytes, oracle.ll128_pack,
              oracle.ll128_unpack),
}


@pytest.fixture(scope="module", autouse=True)
def _init():
    import torch

    torch.cuda.set_device(0)
    rra.rra_init(0)
    rra.rra_set_timeout_ns(2_000_000_000)
    yield


def _dev_bytes(a: np.ndarray):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).copy()).cuda()


def _wire_buf(nbytes):
    import torch

    return torch.full((nbytes,), 0xEE, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("fmt", list(FMT))
@pytest.mark.parametrize("B", [2, 4, 6, 12, 16, 20, 118, 120, 122, 240, 480, 484, 1000, 1024, 4096,
                               65536 + 4, 1 << 20])
def test_pack_bytes_match_oracle(fmt, B):
    pack, _, wire_bytes, opack, _ = FMT[fmt]
    rng = np.random.default_rng(B)
    payload = rng.integers(0, 256, size=B, dtype=np.uint8)
    assert wire_bytes(B) == (oracle.ll_wire_bytes(B) if fmt == "ll" else oracle.ll128_wire_bytes(B))
    wire = _wire_buf(wire_bytes(B))
    pack(_dev_bytes(payload), wire, 0x1234567 if fmt == "ll" else 0x0123456789ABCDEF)
    assert rra.rra_query_status()[0] == 0
    want = opack(payload, 0x1234567 if fmt == "ll" else 0x0123456789ABCDEF)
    assert wire.cpu().numpy().tobytes() == want.tobytes()


@pytest.mark.parametrize("B", [(64 << 20) - 480, 64 << 20, (64 << 20) + 484, (100 << 20) + 6])
def test_ll128_pack_large_payloads(B):
    # from 64 MiB the LL128 pack runs on a grid covering the payload (eight
    # quads a warp in one trip), below it on a resident grid-stride grid
    pack, _, wire_bytes, opack, _ = FMT["ll128"]
    payload = np.random.default_rng(B).integers(0, 256, size=B, dtype=np.uint8)
    wire = _wire_buf(wire_bytes(B))
    pack(_dev_bytes(payload), wire, 0x0F0E0D0C0B0A0908)
    assert rra.rra_query_status()[0] == 0
    assert wire.cpu().numpy().tobytes() == opack(payload, 0x0F0E0D0C0B0A0908).tobytes()


@pytest.mark.parametrize("fmt", list(FMT))
def test_pack_unaligned_payload(fmt):
    import torch

    pack, _, wire_bytes, opack, _ = FMT[fmt]
    B = 4001 * 4
    payload = np.random.default_rng(1).integers(0, 256, size=B + 4, dtype=np.uint8)
    dev = _dev_bytes(payload)
    wire = _wire_buf(wire_bytes(B))
    pack(dev[4:], wire, 9, payload_bytes=B)
    assert rra.rra_query_status()[0] == 0
    assert wire.cpu().numpy().tobytes() == opack(payload[4:], 9).tobytes()


@pytest.mark.parametrize("fmt", list(FMT))
@pytest.mark.parametrize("dtype", ["int32", "float32", "bfloat16"])
@pytest.mark.parametrize("nsrc", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("B", [4, 8, 120, 124, 1000, 4096, 123_456, 1 << 20])
def test_unpack_reduce_matches_oracle(fmt, dtype, nsrc, B):
    import gpu_util as g

    pack, unpack, wire_bytes, opack, ounpack = FMT[fmt]
    e = inputs.ELEM_SIZE[dtype]
    if B % e:
        pytest.skip("whole elements only")
    dist = "int20" if dtype == "int32" else "normal"
    xs = inputs.make_ranks(nsrc, B // e, dtype, dist, seed=B + nsrc)
    wires = []
    for x in xs:
        w = _wire_buf(wire_bytes(B))
        pack(g.to_dev(x, dtype), w, 3)
        wires.append(w)
    out = g.empty(1, B // e, dtype)[0]
    unpack(wires, out, 3)
    st, info = rra.rra_query_status()
    assert st == 0, info
    want, bad = ounpack([opack(x, 3) for x in xs], B, dtype, 3)
    assert bad == -1
    g.assert_bits_equal(g.to_host(out, dtype), want, "%s unpack" % fmt)


@pytest.mark.parametrize("fmt", list(FMT))
def test_ll_config_int32_nsrc4(fmt):
    # n=4 int32 payloads in [-2^20, 2^20], flag = step counter, several steps
    import gpu_util as g

    pack, unpack, wire_bytes, opack, ounpack = FMT[fmt]
    B = 1 << 22
    xs = inputs.cfg_ll_payloads(B)
    wires = [_wire_buf(wire_bytes(B)) for _ in xs]
    devs = [g.to_dev(x, "int32") for x in xs]
    want = np.zeros(B // 4, np.int64)
    for x in xs:
        want += x
    for step in (1, 2, 3):
        for d, w in zip(devs, wires):
            pack(d, w, step)
        out = g.empty(1, B // 4, "int32")[0]
        unpack(wires, out, step)
        assert rra.rra_query_status()[0] == 0
        assert np.array_equal(g.to_host(out, "int32"), want.astype(np.int32))


@pytest.mark.parametrize("fmt", list(FMT))
def test_stale_flag_times_out_and_names_the_line(fmt):
    import gpu_util as g

    pack, unpack, wire_bytes, _, _ = FMT[fmt]
    B = 4 * 10_000
    xs = inputs.cfg_ll_payloads(B)
    wires = []
    for x in xs:
        w = _wire_buf(wire_bytes(B))
        pack(g.to_dev(x, "int32"), w, 5)
        wires.append(w)
    rra.rra_set_timeout_ns(2_000_000)  # 2 ms
    try:
        # corrupt the flag of one line of source 2 from the host
        line, flag_off = (8, 4) if fmt == "ll" else (128, 120)
        bad_line = 1234 if fmt == "ll" else 77
        wires[2][bad_line * line + flag_off] ^= 0x40
        out = g.empty(1, B // 4, "int32")[0]
        unpack(wires, out, 5)
        st, info = rra.rra_query_status()
        assert st == rra.RRA_ERR_TIMEOUT
        assert info[0] == rra.RRA_ERR_TIMEOUT and info[1] == 2 and info[3] == bad_line
        # the GPU is still usable: a call one step late times out at line 0 ...
        wires[2][bad_line * line + flag_off] ^= 0x40
        unpack(wires, out, 6)
        st, info = rra.rra_query_status()
        assert st == rra.RRA_ERR_TIMEOUT
        # ... and the right step succeeds
        unpack(wires, out, 5)
        assert rra.rra_query_status()[0] == 0
    finally:
        rra.rra_set_timeout_ns(2_000_000_000)
