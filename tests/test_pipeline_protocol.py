"""Models of the tensor-core kernels' mbarrier protocols, run under random schedules.

Each role of a kernel (producers, converter warps, MMA issuers, softmax warps) is a sequence of
waits on, and arrivals at, the kernel's mbarriers in the order the CUDA source issues them; the asynchronous arrivals (TMA copies landing, tcgen05.commit)
happen at random later moments. An mbarrier wait names a phase by its parity only, so the
protocol is correct only if every wait for phase k starts when the barrier has completed k or
k + 1 phases and no barrier completes phase k + 2 while a wait for phase k is still pending.
The tests check that, and that every schedule runs to its end, for 1 to 12 tiles per item, for
the widening kernel, the FP8 kernel and the 16-bit few-row kernel (softmax warps modelled one by
one, so that a fast warp can run ahead of a slow one); and that the check catches planted
mistakes.
"""
import random

import pytest

SK, SV = 2, 3          # staging ring depths: K, V


class Bar:
    def __init__(self, name, count=1):
        self.name, self.done, self.count, self.pending = name, 0, count, 0

    def arrive(self, waits):
        self.pending += 1
        if self.pending < self.count:
            return
        self.pending = 0
        for (bar, k, who) in waits:
            if bar is self and k < self.done:
                raise AssertionError(f"{self.name}: phase {self.done} completes while {who} still waits phase {k}")
        self.done += 1


def roles(n, rnd, rescale_p, skip_v_wait=False, sk=SK, sv=SV, nk16=2, v_wait_at_v=False):
    """The widening kernel: staging rings of depth sk (K) and sv (V), nk16 f16 K buffers; with
    v_wait_at_v the converters wait for a staged V tile when they widen it instead of before
    widening the K tile of the same index (the 16-bit caches, which read no V scales)."""
    def prod(name, depth):
        for j in range(n):
            st = j % depth
            if j >= depth:
                yield ("wait", f"e{name}8{st}", j // depth - 1)
            yield ("async", [f"f{name}8{st}"])
        for j in range(max(0, n - depth), n):
            yield ("wait", f"f{name}8{j % depth}", j // depth)

    def conv():
        for step in range(n + 1):
            if step < n:
                j = step
                yield ("wait", f"fK8{j % sk}", j // sk)
                if not v_wait_at_v:
                    yield ("wait", f"fV8{j % sv}", j // sv)
                yield ("arrive", f"meta{j % 4}")
                if j >= nk16:
                    yield ("wait", f"eK16{j % nk16}", j // nk16 - 1)
                yield ("arrive", f"fK16{j % nk16}")
                yield ("arrive", f"eK8{j % sk}")
            if step >= 1:
                j = step - 1
                if v_wait_at_v:
                    yield ("wait", f"fV8{j % sv}", j // sv)
                if j >= 1 and not skip_v_wait:
                    yield ("wait", "eV16", j - 1)
                yield ("arrive", "fV16")
                yield ("arrive", f"eV8{j % sv}")
        for j in range(max(0, n - nk16), n):
            yield ("wait", f"eK16{j % nk16}", j // nk16)
        yield ("wait", "eV16", n - 1)

    def qk():
        yield ("wait", "q", 0)
        for j in range(n):
            yield ("wait", f"fK16{j % nk16}", j // nk16)
            if j >= 2:
                yield ("wait", f"sfree{j & 1}", (j >> 1) - 1)
            yield ("async", [f"sfull{j & 1}", f"eK16{j % nk16}"])

    def pv():
        for j in range(n):
            yield ("wait", f"pfull{j & 1}", j >> 1)
            yield ("wait", "fV16", j)
            yield ("async", [f"pv{j & 1}", "eV16"])

    def soft():
        yield ("arrive", "q")
        last = -1
        for j in range(n):
            last = j
            yield ("wait", f"meta{j % 4}", j >> 2)
            yield ("wait", f"sfull{j & 1}", j >> 1)
            yield ("arrive", f"sfree{j & 1}")
            if j >= 2:
                yield ("wait", f"pv{j & 1}", (j >> 1) - 1)
            if j >= 1 and rnd.random() < rescale_p:       # the O rescale waits for the last PV
                yield ("wait", f"pv{(j - 1) & 1}", (j - 1) >> 1)
            yield ("arrive", f"pfull{j & 1}")
        if last >= 1:
            yield ("wait", f"pv{(last - 1) & 1}", (last - 1) >> 1)
        if last >= 0:
            yield ("wait", f"pv{last & 1}", last >> 1)

    return {"prodK": prod("K", sk), "prodV": prod("V", sv), "conv": conv(), "qk": qk(), "pv": pv(),
            "soft": soft()}


SM_WARPS = 2          # softmax warps modelled per warpgroup (the kernel has 8)
FP8_STAGES = 4
FP8_COUNTS = {"sfree": SM_WARPS, "pfull": SM_WARPS, "xmax": SM_WARPS, "q": SM_WARPS, "fin": 2}


def fp8_roles(n, rnd, partial_p, skip_p_wait=False):
    """The FP8 kernel: K and V producers (4-stage rings, two tiles per step), the QK^T and PV
    issuers, and two softmax warpgroups taking tiles wg, wg + 2, ... with their own S buffer,
    P buffer and row-maximum barrier (split phase: arrive, work, wait)."""
    def prod(name):
        for j0 in range(0, n, 2):
            for j in range(j0, min(n, j0 + 2)):
                if j >= FP8_STAGES:
                    yield ("wait", f"{name}empty{j % FP8_STAGES}", j // FP8_STAGES - 1)
            for j in range(j0, min(n, j0 + 2)):
                yield ("async", [f"{name}full{j % FP8_STAGES}"])
        for j in range(max(0, n - FP8_STAGES), n):
            yield ("wait", f"{name}full{j % FP8_STAGES}", j // FP8_STAGES)
        for j in range(max(0, n - FP8_STAGES), n):
            yield ("wait", f"{name}empty{j % FP8_STAGES}", j // FP8_STAGES)

    def qk():
        yield ("wait", "q", 0)
        for j in range(n):
            yield ("wait", f"kfull{j % FP8_STAGES}", j // FP8_STAGES)
            if j >= 2:
                yield ("wait", f"sfree{j & 1}", (j >> 1) - 1)
            yield ("async", [f"sfull{j & 1}", f"kempty{j % FP8_STAGES}"])
        yield ("async", ["fin"])
        yield ("wait", "fin", 0)

    def pv():
        for j in range(n):
            yield ("wait", f"pfull{j & 1}", j >> 1)
            yield ("wait", f"vfull{j % FP8_STAGES}", j // FP8_STAGES)
            yield ("async", [f"pv{j & 1}", f"vempty{j % FP8_STAGES}"])
        yield ("async", ["fin"])
        yield ("wait", "fin", 0)

    def soft(wg, duty):
        if wg == 0:
            yield ("arrive", "q")
        else:
            yield ("wait", "q", 0)
        last = -1
        for j in range(wg, n, 2):
            last = j
            yield ("wait", f"sfull{wg}", j >> 1)
            if duty and rnd.random() < partial_p:           # a partial tile: its V rows are zeroed
                yield ("wait", f"vfull{j % FP8_STAGES}", j // FP8_STAGES)
            yield ("arrive", f"sfree{wg}")
            yield ("arrive", f"xmax{wg}")
            yield ("wait", f"xmax{wg}", j >> 1)
            if j >= 2 and not skip_p_wait:
                yield ("wait", f"pv{wg}", (j - 2) >> 1)
            yield ("arrive", f"pfull{wg}")
        if last >= 0:
            yield ("wait", f"pv{wg}", last >> 1)

    actors = {"prodK": prod("k"), "prodV": prod("v"), "qk": qk(), "pv": pv()}
    for wg in range(2):
        for w in range(SM_WARPS):
            actors[f"soft{wg}.{w}"] = soft(wg, duty=w == 0)
    return actors


B16_STAGES = 3
B16_COUNTS = {"sfree": SM_WARPS, "pfull": SM_WARPS, "q": SM_WARPS, "fin": 2}


def b16_roles(n, rnd, p_rare):
    """The 16-bit few-row kernel: K and V producers (3-stage rings), the S^T and O^T issuers,
    and one softmax group of warps taking every tile (two S and two P buffers)."""
    def prod(name):
        for j in range(n):
            if j >= B16_STAGES:
                yield ("wait", f"{name}empty{j % B16_STAGES}", j // B16_STAGES - 1)
            yield ("async", [f"{name}full{j % B16_STAGES}"])
        for j in range(max(0, n - B16_STAGES), n):
            yield ("wait", f"{name}full{j % B16_STAGES}", j // B16_STAGES)
        for j in range(max(0, n - B16_STAGES), n):
            yield ("wait", f"{name}empty{j % B16_STAGES}", j // B16_STAGES)

    def qk():
        yield ("wait", "q", 0)
        for j in range(n):
            yield ("wait", f"kfull{j % B16_STAGES}", j // B16_STAGES)
            if j >= 2:
                yield ("wait", f"sfree{j & 1}", (j >> 1) - 1)
            yield ("async", [f"sfull{j & 1}", f"kempty{j % B16_STAGES}"])
        yield ("async", ["fin"])
        yield ("wait", "fin", 0)

    def pv():
        for j in range(n):
            yield ("wait", f"pfull{j & 1}", j >> 1)
            yield ("wait", f"vfull{j % B16_STAGES}", j // B16_STAGES)
            yield ("async", [f"pv{j & 1}", f"vempty{j % B16_STAGES}"])
        yield ("async", ["fin"])
        yield ("wait", "fin", 0)

    def soft():
        yield ("arrive", "q")
        for j in range(n):
            yield ("wait", f"sfull{j & 1}", j >> 1)
            if rnd.random() < p_rare:                      # a token not read: its V rows are zeroed
                yield ("wait", f"vfull{j % B16_STAGES}", j // B16_STAGES)
            yield ("arrive", f"sfree{j & 1}")
            if j >= 2:
                yield ("wait", f"pv{j & 1}", (j - 2) >> 1)
            if j >= 1 and rnd.random() < p_rare:          # the reference moved: O is rescaled
                yield ("wait", f"pv{(j - 1) & 1}", (j - 1) >> 1)
            yield ("arrive", f"pfull{j & 1}")
        yield ("wait", f"pv{(n - 1) & 1}", (n - 1) >> 1)

    actors = {"prodK": prod("k"), "prodV": prod("v"), "qk": qk(), "pv": pv()}
    for w in range(SM_WARPS):
        actors[f"soft{w}"] = soft()
    return actors


def run(n, seed, rescale_p=0.3, skip_v_wait=False, model="widening", skip_p_wait=False, **shape):
    rnd = random.Random(seed)
    bars = {}
    counts = {"fp8": FP8_COUNTS, "b16": B16_COUNTS}.get(model, {})

    def bar(name):
        if name not in bars:
            bars[name] = Bar(name, counts.get(name.rstrip("0123456789"), 1))
        return bars[name]

    if model == "widening":
        actors = roles(n, rnd, rescale_p, skip_v_wait, **shape)
    elif model == "fp8":
        actors = fp8_roles(n, rnd, rescale_p, skip_p_wait)
    else:
        actors = b16_roles(n, rnd, rescale_p)
    cur = {k: next(g, None) for k, g in actors.items()}
    pending = []
    for _ in range(200000):
        waits = [(bar(a[1]), a[2], k) for k, a in cur.items() if a and a[0] == "wait"]
        ready = [k for k, a in cur.items() if a is not None and (a[0] != "wait" or bar(a[1]).done > a[2])]
        choices = ready + (["async"] if pending else [])
        if not choices:
            assert all(a is None for a in cur.values()), f"deadlock with {n} tiles: {cur}"
            return
        c = rnd.choice(choices)
        if c == "async":
            bar(pending.pop(rnd.randrange(len(pending)))).arrive(waits)
            continue
        a = cur[c]
        if a[0] == "wait":
            assert bar(a[1]).done <= a[2] + 1, f"{c} waits {a[1]} phase {a[2]} after {bar(a[1]).done} phases"
        elif a[0] == "arrive":
            bar(a[1]).arrive(waits)
        else:
            pending.extend(a[1])
        cur[c] = next(actors[c], None)
        nxt = cur[c]
        if nxt is not None and nxt[0] == "wait":
            assert bar(nxt[1]).done >= nxt[2], f"{c} waits {nxt[1]} phase {nxt[2]} before phase {nxt[2] - 1} completed"
    raise AssertionError("schedule did not end")


@pytest.mark.parametrize("n", list(range(1, 13)))
def test_widening_kernel_barrier_protocol(n):
    for seed in range(100):
        run(n, 7919 * n + seed)


def test_the_protocol_check_catches_a_missing_wait():
    """Widening V without waiting for the previous PV lets the V buffer's barrier run two
    phases ahead of the PV issuer's wait."""
    with pytest.raises(AssertionError):
        for seed in range(200):
            run(6, seed, skip_v_wait=True)


@pytest.mark.parametrize("n", list(range(1, 13)))
def test_fp8_kernel_barrier_protocol(n):
    for seed in range(100):
        run(n, 104729 * n + seed, model="fp8")


def test_the_fp8_protocol_check_catches_a_missing_wait():
    """Writing P without waiting for the PV that read the buffer two tiles before lets the P
    buffer's barrier run ahead of the PV issuer."""
    with pytest.raises(AssertionError):
        for n in range(3, 9):
            for seed in range(200):
                run(n, seed, model="fp8", skip_p_wait=True)


@pytest.mark.parametrize("n", list(range(1, 13)))
def test_sixteen_bit_kernel_barrier_protocol(n):
    for seed in range(100):
        run(n, 15485863 * n + seed, model="b16")


@pytest.mark.parametrize("nk16", [1, 2])
@pytest.mark.parametrize("n", list(range(1, 13)))
def test_widening_kernel_one_deep_rings(n, nk16):
    """The 16-bit head_dim-256 instance of the widening kernel: one-deep K and V staging rings,
    one or two f16 K buffers, and the staged V tile waited for when it is widened."""
    for seed in range(60):
        run(n, 104729 * n + seed, sk=1, sv=1, nk16=nk16, v_wait_at_v=True)


def test_one_deep_v_ring_needs_the_v_wait_at_v():
    """Waiting for V(j) before widening K(j), as the deeper rings do, deadlocks a one-deep V
    ring: V(j) cannot land before V(j - 1) is widened, which comes after K(j)."""
    with pytest.raises(AssertionError, match="deadlock"):
        for seed in range(50):
            run(3, seed, sk=1, sv=1, nk16=1, v_wait_at_v=False)
