"""The gathered-expert MLP (tinfer_op_moe): the two fixed-shape kernels that read the chosen
experts' weights through a device index tensor ("One launch per token", "The same trick, sparser: a
64-expert MoE"), against the oracle's orc_moe_mlp on the same seeded weights, ids and routing
weights."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import decode_persistent_megakernel_gb300 as T  # noqa: E402
import synth  # noqa: E402
from oracle import Oracle  # noqa: E402

pytestmark = pytest.mark.gpu
ORC = Oracle("f64")


def dev(a):
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
    return t.cuda()


class Moe:
    """A packed gathered-expert case on the GPU."""

    def __init__(self, m, fmt, group, sdt):
        self.m, self.fmt, self.group, self.sdt = m, fmt, group, sdt
        self.f = T.TINFER_INT4 if fmt == "int4" else T.TINFER_BF16
        self.sd_code = T.TINFER_SCALE_BF16 if sdt == "bf16" else T.TINFER_SCALE_FP16
        self.E, self.F, self.H = m["wg"].shape[0], m["wg"].shape[1], m["wd"].shape[1]
        keep = {k: dev(v) for k, v in m.items() if v is not None and k[0] in "ws" and k != "weights"}
        self.keep = keep
        nb = [T.tinfer_moe_packed_bytes(self.f, group, self.E, self.H, self.F, w) for w in (0, 1)]
        assert min(nb) > 0
        self.gu = torch.empty(nb[0], dtype=torch.uint8, device="cuda")
        self.down = torch.empty(nb[1], dtype=torch.uint8, device="cuda")
        assert T.tinfer_pack_moe(self.f, group, self.sd_code, self.E, self.H, self.F, keep["wg"], keep.get("sg"),
                                 keep["wu"], keep.get("su"), keep["wd"], keep.get("sd"), self.gu, self.down) == 0

    def run(self, ids, weights, x, y=None, accumulate=0, status=None):
        k = len(ids)
        ids_d = torch.tensor(np.asarray(ids, np.int32), device="cuda")
        w_d = torch.tensor(np.asarray(weights, np.float32), device="cuda")
        x_d = torch.tensor(np.asarray(x, np.float32), device="cuda")
        h = torch.empty(k * self.F, dtype=torch.float32, device="cuda")
        if y is None:
            y = torch.empty(self.H, dtype=torch.float32, device="cuda")
        rc = T.tinfer_op_moe(self.f, self.group, self.sd_code, self.E, k, self.H, self.F, self.gu, self.down,
                             ids_d, w_d, x_d, h, y, accumulate, status)
        assert rc == 0
        torch.cuda.synchronize()
        return y.cpu().numpy().astype(np.float64)

    def ref(self, ids, weights, x):
        m = self.m
        return ORC.moe_mlp(self.f, self.group, self.sdt == "bf16", m["wg"], m["sg"], m["wu"], m["su"], m["wd"],
                           m["sd"], np.asarray(ids, np.int32), np.asarray(weights, np.float64),
                           np.asarray(x, np.float64))


def check(got, ref):
    # fp32 accumulation against fp64: relative to the output's scale
    scale = float(np.abs(ref).max())
    np.testing.assert_allclose(got, ref, rtol=1e-4, atol=1e-5 * scale)


@pytest.mark.parametrize("fmt,group,sdt", [("bf16", 64, "fp16"), ("int4", 64, "fp16"), ("int4", 128, "bf16")])
@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_moe_small_matches_oracle(fmt, group, sdt, k):
    m = synth.make_moe(16, k, 512, 256, fmt, group, sdt, seed=k)
    moe = Moe(m, fmt, group, sdt)
    check(moe.run(m["ids"], m["weights"], m["x"]), moe.ref(m["ids"], m["weights"], m["x"]))


@pytest.mark.parametrize("fmt,group,sdt", [("bf16", 64, "fp16"), ("int4", 64, "fp16")])
def test_moe_64_experts_top8_full_size(fmt, group, sdt):
    # OLMoE-like synthetic shape: 64 experts, 8 chosen, hidden 2048, expert FFN 1024
    m = synth.make_moe(64, 8, 2048, 1024, fmt, group, sdt, seed=0)
    moe = Moe(m, fmt, group, sdt)
    y1 = moe.run(m["ids"], m["weights"], m["x"])
    check(y1, moe.ref(m["ids"], m["weights"], m["x"]))
    # the same ids in another order with their weights: the same experts, summed in another order
    perm = np.array([3, 1, 7, 0, 6, 2, 5, 4])
    check(moe.run(m["ids"][perm], m["weights"][perm], m["x"]), moe.ref(m["ids"], m["weights"], m["x"]))
    # fixed-shape reuse: a second routing through the same packed experts, and reproducibility
    ids2 = np.array([(int(e) + 9) % 64 for e in m["ids"]], np.int32)
    check(moe.run(ids2, m["weights"], m["x"]), moe.ref(ids2, m["weights"], m["x"]))
    assert np.array_equal(moe.run(m["ids"], m["weights"], m["x"]), y1)


def test_moe_accumulates_and_reports_bad_ids():
    m = synth.make_moe(16, 4, 512, 256, "bf16", seed=7)
    moe = Moe(m, "bf16", 64, "fp16")
    y0 = np.linspace(-1, 1, 512).astype(np.float32)
    y = torch.tensor(y0, device="cuda")
    got = moe.run(m["ids"], m["weights"], m["x"], y=y, accumulate=1)
    check(got - y0, moe.ref(m["ids"], m["weights"], m["x"]))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = m["ids"].copy()
    bad[2] = 99  # outside [0, 16): read as expert 0 and reported
    got = moe.run(bad, m["weights"], m["x"], status=status)
    assert int(status.item()) == 1
    fixed = bad.copy()
    fixed[2] = 0
    check(got, moe.ref(fixed, m["weights"], m["x"]))
    status.zero_()
    moe.run(m["ids"], m["weights"], m["x"], status=status)
    assert int(status.item()) == 0


def test_moe_host_validation():
    m = synth.make_moe(16, 4, 512, 256, "bf16", seed=8)
    moe = Moe(m, "bf16", 64, "fp16")
    x = torch.zeros(512, device="cuda")
    h = torch.empty(3 * 256, device="cuda")
    y = torch.empty(512, device="cuda")
    ids = torch.zeros(3, dtype=torch.int32, device="cuda")
    w = torch.zeros(3, device="cuda")
    # top_k must divide the eight consumer warps
    assert T.tinfer_op_moe(0, 64, 0, 16, 3, 512, 256, moe.gu, moe.down, ids, w, x, h, y) == T.TINFER_ERR_UNSUPPORTED
    assert T.tinfer_op_moe(0, 64, 0, 16, 4, 512, 256, moe.gu, moe.down, ids, w, None, h, y) == T.TINFER_ERR_INVALID_ARG
    assert T.tinfer_moe_packed_bytes(1, 48, 16, 512, 256, 0) == 0  # group not a multiple of 32
