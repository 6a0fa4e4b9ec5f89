"""Seeded single-fault checks of every compute entry point's argument
validation (qgZ, qwZ, SR).

Each case starts from a random valid geometry (R, G | R, B, k blocks per
shard; or n and B) with placeholder pointers and breaks exactly one
documented rule --
a geometry rule, a required pointer left NULL or misaligned, an optional
pointer misaligned, one of a both-or-neither pair missing, a bad output type,
a block too small for the fused kernels -- and expects that rule's status
code, with the entry point named in wc_last_error().  Every call breaks a
rule, so none reaches a launch; the file still runs only where no GPU is
visible, since its pointers are placeholders."""
import random

import pytest

from weight_communication_gb300 import binding

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="placeholder pointers: run where no GPU is reachable")

from test_abi import FAKE, MIS, lib  # noqa: E402,F401  (the library fixture)

EINVAL, EALIGN, ERANGE = binding.WC_EINVAL, binding.WC_EALIGN, binding.WC_ERANGE

# Entry point: parameter names in order, and which pointers are required
# (NULL and misalignment refused), optional (misalignment refused), or a
# both-or-neither pair.  "G" absent means the call fixes G = 1.
ENTRIES = {
    "wc_ef_quant_int4": (["g", "ef", "codes", "scales", "N", "R", "G", "B", "s", "beta", "st"],
                         ["g", "codes", "scales"], ["ef"], None),
    "wc_ef_quant_int4_bf16ef": (["g", "ef", "codes", "scales", "N", "R", "G", "B", "s", "beta",
                                 "st"], ["g", "ef", "codes", "scales"], [], None),
    "wc_ef_quant_int4_int8ef": (["g", "ef", "es", "codes", "scales", "N", "R", "G", "B", "s",
                                 "beta", "st"], ["g", "ef", "es", "codes", "scales"], [], None),
    "wc_dequant_reduce": (["codes", "scales", "N", "R", "G", "B", "os", "out", "dt", "st"],
                          ["codes", "scales", "out"], [], None),
    "wc_dequant_reduce_requant": (["codes", "scales", "N", "R", "G", "B", "oc", "osc", "st"],
                                  ["codes", "scales", "oc", "osc"], [], None),
    "wc_dequant_reduce_requant_ef": (["codes", "scales", "N", "R", "G", "B", "oc", "osc", "ef1",
                                      "s", "beta", "st"],
                                     ["codes", "scales", "oc", "osc", "ef1"], [], None),
    "wc_qgz_step_fused": (["g", "ef", "codes", "scales", "N", "R", "B", "s", "beta", "os", "out",
                           "dt", "st"], ["g", "out"], ["ef"], ("codes", "scales")),
    "wc_qgz_step_fused_bf16ef": (["g", "ef", "codes", "scales", "N", "R", "B", "s", "beta", "os",
                                  "out", "dt", "st"], ["g", "ef", "out"], [], ("codes", "scales")),
    "wc_qgz_step_fused_int8ef": (["g", "ef", "es", "codes", "scales", "N", "R", "B", "s", "beta",
                                  "os", "out", "dt", "st"], ["g", "ef", "es", "out"], [],
                                 ("codes", "scales")),
    "wc_qgz_first_hop_fused": (["g", "ef", "codes", "scales", "N", "R", "G", "B", "s", "beta",
                                "oc", "osc", "ef1", "st"], ["g", "oc", "osc"], ["ef", "ef1"],
                               ("codes", "scales")),
    "wc_qgz_first_hop_fused_bf16ef": (["g", "ef", "codes", "scales", "N", "R", "G", "B", "s",
                                       "beta", "oc", "osc", "ef1", "st"],
                                      ["g", "ef", "oc", "osc"], ["ef1"], ("codes", "scales")),
    "wc_qgz_first_hop_fused_int8ef": (["g", "ef", "es", "codes", "scales", "N", "R", "G", "B",
                                       "s", "beta", "oc", "osc", "ef1", "st"],
                                      ["g", "ef", "es", "oc", "osc"], ["ef1"],
                                      ("codes", "scales")),
}
FUSED = {n for n in ENTRIES if "fused" in n}
WITH_DTYPE = {n for n in ENTRIES if "dt" in ENTRIES[n][0]}


def valid_args(name: str, rng: random.Random) -> dict:
    names = ENTRIES[name][0]
    R = rng.choice([1, 2, 3, 4, 6, 8, 12, 16, 32, 48])
    G = rng.choice([d for d in range(1, R + 1) if R % d == 0]) if "G" in names else 1
    B = rng.choice([128, 256, 512, 1024] if name in FUSED else [32, 64, 128, 256, 512, 1024])
    N = R * B * rng.randint(1, 7)
    a = {n: FAKE for n in names}
    a.update(N=N, R=R, G=G, B=B, s=1.0, beta=0.5, os=1.0, dt=binding.WC_F32, st=None)
    return {n: a[n] for n in names}


def faults(name: str, a: dict, rng: random.Random):
    """(description, changed arguments, expected status) for one rule each."""
    names, required, optional, pair = ENTRIES[name]
    R, B = a["R"], a["B"]
    out = [("negative N", {"N": -R * B}, EINVAL),
           ("R = 0", {"R": 0}, EINVAL),
           ("B not a power of two in [32, 1024]",
            {"B": rng.choice([0, 16, 24, 48, 96, 1000, 2048, 4096])}, EINVAL),
           ("B does not divide N/R", {"N": R * (B * rng.randint(1, 5) + B // 2)}, EINVAL),
           ("R*N reaches 2^32", {"R": 2, "G": 1, "B": 256, "N": 1 << 31}, ERANGE)]
    if R >= 2:
        out.append(("R does not divide N", {"N": a["N"] + 1}, EINVAL))
    if "G" in names:
        out += [("G = 0", {"G": 0}, EINVAL), ("G does not divide R", {"G": R + 1}, EINVAL)]
    if name in FUSED:
        out.append(("B below 128", {"B": 64}, EINVAL))
    if name in WITH_DTYPE:
        out.append(("unknown output type", {"dt": rng.choice([-1, 2, 7])}, EINVAL))
    for p in required:
        out += [(f"{p} NULL", {p: None}, EINVAL), (f"{p} misaligned", {p: MIS}, EALIGN)]
    for p in optional:
        out.append((f"{p} misaligned", {p: MIS}, EALIGN))
    if pair:
        out += [(f"{pair[0]} without {pair[1]}", {pair[1]: None}, EINVAL),
                (f"{pair[1]} without {pair[0]}", {pair[0]: None}, EINVAL),
                (f"{pair[0]} misaligned", {pair[0]: MIS}, EALIGN)]
    return out


@pytest.mark.parametrize("name", sorted(ENTRIES))
def test_every_single_fault_is_refused(lib, name):
    rng = random.Random(sum(map(ord, name)))
    f = getattr(lib, name)
    checked = 0
    for _ in range(60):
        a = valid_args(name, rng)
        for what, change, want in faults(name, a, rng):
            args = dict(a, **change)
            rc = f(*args.values())
            assert rc == want, (name, what, args, rc, lib.wc_last_error())
            msg = lib.wc_last_error().decode()
            assert name in msg, (name, what, msg)
            checked += 1
    assert checked > 500


# qwZ and SR: parameter names, required pointers.
SIZE_ENTRIES = {
    "wc_qwz_quant_int8": (["w", "codes", "scales", "n", "B", "st"], ["w", "codes", "scales"]),
    "wc_qwz_quant_replica_int8": (["w", "codes", "scales", "rep", "n", "B", "st"],
                                  ["w", "codes", "scales", "rep"]),
    "wc_qwz_dequant_int8": (["codes", "scales", "out", "n", "B", "st"],
                            ["codes", "scales", "out"]),
    "wc_sr_accumulate_bf16": (["dst", "src", "n", "seed", "step", "st"], ["dst", "src"]),
}


def size_faults(name: str, rng: random.Random):
    names, required = SIZE_ENTRIES[name]
    if name.startswith("wc_qwz"):
        B = 32 << rng.randint(0, 7)
        a = dict.fromkeys(names, FAKE)
        a.update(n=B * rng.randint(1, 4096), B=B, st=None)
        out = [("negative n", {"n": -B}, EINVAL),
               ("B not a power of two in [32, 4096]",
                {"B": rng.choice([0, 16, 48, 100, 8192])}, EINVAL),
               ("B does not divide n", {"n": a["n"] + B // 2}, EINVAL),
               ("n reaches 2^32", {"n": 1 << 32, "B": 2048}, ERANGE)]
    else:
        n = rng.randint(1, 1 << 20)
        a = {"dst": FAKE, "src": FAKE + ((2 * n + 15) // 16) * 16 + 16, "n": n,
             "seed": rng.getrandbits(32), "step": rng.randint(0, 7), "st": None}
        out = [("negative n", {"n": -1}, EINVAL),
               ("n reaches 2^32", {"n": 1 << 32}, ERANGE),
               ("dst and src overlap", {"src": FAKE + 16, "n": max(n, 9)}, EINVAL)]
    for p in required:
        out += [(f"{p} NULL", {p: None}, EINVAL), (f"{p} misaligned", {p: MIS}, EALIGN)]
    return {k: a[k] for k in names}, out


@pytest.mark.parametrize("name", sorted(SIZE_ENTRIES))
def test_every_single_size_fault_is_refused(lib, name):
    rng = random.Random(sum(map(ord, name)))
    f = getattr(lib, name)
    checked = 0
    for _ in range(60):
        a, cases = size_faults(name, rng)
        for what, change, want in cases:
            args = dict(a, **change)
            rc = f(*args.values())
            assert rc == want, (name, what, args, rc, lib.wc_last_error())
            assert name in lib.wc_last_error().decode(), (name, what)
            checked += 1
    assert checked > 300
