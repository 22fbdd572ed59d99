"""Model check of the single-token kernels' cross-block protocol
(bit_expert_matvec_moe_b300/csrc/moe_decode_b1.cu: decode_b1_kernel, one layer a
launch, and decode_stack_kernel, several layers a launch) on a shared
workspace: the blocks of a launch are coroutines interleaved at random, each
step one load, store or atomic of the kernel's protocol:

  start       n = atomicAdd(launches, 1); the first layer's epoch = n / P + 1;
              (stack) read the output-row counter's base
  each layer  (stack, l > 0) wait until the output-row counter reaches
              base + P * l, read every block's output word of layer l - 1;
              publish the logit word, add to the logit counter, poll every
              block's logit word; publish the activation word, add to the
              activation counter, wait until it reaches P * epoch, read every
              block's activation word; (stack, not the last layer) publish the
              output word and add to the output-row counter
  end         (stack) add L - 1 to the launch counter
  failure     a wait that runs out sets abort; every block then leaves through
              the cleanup, which adds the epoch counters it still owes for this
              and the later layers and, for a stack, the L - 1 launches

Every published word carries (epoch, launch, layer).  A reader accepts a word
only when its epoch is the one it expects, so the check is: whenever a word is
accepted, it was written by the same launch for the same layer (epochs never
collide across launches and layers, single-layer and stack launches mixed), and
every launch without an injected failure completes (no wait is left without
its writers).  After a failed launch the error state is cleared, as by
moe_get_device_status, and later launches must again complete."""
import random

import pytest


class Ws:
    def __init__(s, P):
        s.P = P
        s.launches = s.pub_lg_cnt = s.pub_act_cnt = s.pub_h_cnt = 0
        s.abort = False
        s.status = 0
        s.hook = 0
        s.lg = [(0, None)] * P
        s.act = [(0, None)] * P
        s.h = [(0, None)] * P


def block(ws, b, launch_id, L, stack, fail_at, budget, mutate=None):
    """One block's protocol steps as a generator (each yield: one step or a
    wait that is not yet satisfied).  fail_at: the index of the wait at which
    this block gives up (None: never).  mutate plants a protocol mistake for
    the test that the model catches it: "same_epoch" (every layer of a launch
    uses its first epoch), "no_launch_tail" (a stack launch does not add its
    further layers to the launch counter).  Returns via StopIteration."""
    P = ws.P
    waits = [0]

    def wait(cond):
        # a bounded wait: gives up on abort, on the injected failure, or when
        # the step budget runs out (the model's 1 s)
        k = waits[0]
        waits[0] += 1
        spent = 0
        while True:
            if ws.abort:
                return False
            if fail_at is not None and k == fail_at:
                ws.abort = True
                ws.status |= 1
                return False
            if cond():
                return True
            spent += 1
            if spent > budget:
                ws.abort = True
                ws.status |= 1
                return False
            yield

    bumped = {"lg": False, "act": False}
    n = ws.launches
    ws.launches += 1
    yield
    base = n // P + 1
    hook = ws.hook
    hbase = ws.pub_h_cnt if stack else 0
    yield
    l = 0
    ok = not ws.abort
    while ok and l < L:
        layer_epoch = 0 if mutate == "same_epoch" else l
        epoch, expect = base + layer_epoch, base + layer_epoch + hook
        bumped = {"lg": False, "act": False}
        tag = (launch_id, l)
        if stack and l > 0:
            ok = yield from wait(lambda: ws.pub_h_cnt >= hbase + P * (l + hook))
            if not ok:
                break
            ok = yield from wait(lambda: all(w[0] == expect - (0 if mutate == "same_epoch" else 1) for w in ws.h))
            if not ok:
                break
            assert all(w[1] == (launch_id, l - 1) for w in ws.h), ("stale output word accepted", ws.h, tag)
        ws.lg[b] = (epoch, tag)
        yield
        ws.pub_lg_cnt += 1
        bumped["lg"] = True
        yield
        ok = yield from wait(lambda: all(w[0] == expect for w in ws.lg))
        if not ok:
            break
        assert all(w[1] == tag for w in ws.lg), ("stale logit word accepted", ws.lg, tag)
        ws.act[b] = (epoch, tag)
        yield
        ws.pub_act_cnt += 1
        bumped["act"] = True
        yield
        ok = yield from wait(lambda: ws.pub_act_cnt >= P * (expect + (l if mutate == "same_epoch" else 0)))
        if not ok:
            break
        ok = yield from wait(lambda: all(w[0] == expect for w in ws.act))
        if not ok:
            break
        assert all(w[1] == tag for w in ws.act), ("stale activation word accepted", ws.act, tag)
        if stack and l + 1 < L:
            ws.h[b] = (epoch, tag)
            yield
            ws.pub_h_cnt += 1
            yield
        l += 1
    if ok:
        if stack and L > 1 and mutate != "no_launch_tail":
            ws.launches += L - 1
        return "done"
    # cleanup: the epoch counters this block still owes, and the launches
    later = L - 1 - l
    ws.pub_lg_cnt += (0 if bumped["lg"] else 1) + later
    ws.pub_act_cnt += (0 if bumped["act"] else 1) + later
    if stack and L > 1:
        ws.launches += L - 1
    return "failed"


def run_launch(ws, rnd, launch_id, L, stack, fail_block=None, fail_at=None, budget=10_000, mutate=None):
    gens = {b: block(ws, b, launch_id, L, stack, fail_at if b == fail_block else None, budget, mutate)
            for b in range(ws.P)}
    results = {}
    while gens:
        b = rnd.choice(list(gens))
        try:
            next(gens[b])
        except StopIteration as e:
            results[b] = e.value
            del gens[b]
    return results


def clear_error_state(ws):
    ws.abort = False
    ws.status = 0
    ws.hook = 0


@pytest.mark.parametrize("seed", range(12))
def test_mixed_single_and_stack_launches_complete_with_their_own_words(seed):
    rnd = random.Random(seed)
    ws = Ws(P=rnd.choice([2, 3, 5]))
    for launch_id in range(14):
        stack = rnd.random() < 0.6
        L = rnd.choice([1, 2, 3, 5]) if stack else 1
        res = run_launch(ws, rnd, launch_id, L, stack)
        assert set(res.values()) == {"done"}, (launch_id, res)
        # every counter stays a whole number of grids per layer-epoch
        assert ws.launches % ws.P == 0 and ws.pub_act_cnt == ws.P * (ws.launches // ws.P)
        assert ws.pub_lg_cnt == ws.pub_act_cnt


@pytest.mark.parametrize("seed", range(12))
def test_failed_launch_leaves_the_workspace_usable(seed):
    rnd = random.Random(100 + seed)
    ws = Ws(P=rnd.choice([2, 3, 4]))
    for launch_id in range(10):
        stack = rnd.random() < 0.7
        L = rnd.choice([1, 2, 4]) if stack else 1
        if launch_id in (3, 6):
            # one block gives up at a random wait (as a bounded wait that ran
            # out): every block must leave, and the counters must stay in step
            res = run_launch(ws, rnd, launch_id, L, stack, fail_block=rnd.randrange(ws.P),
                             fail_at=rnd.randrange(1 + 3 * L))
            assert all(v in ("done", "failed") for v in res.values())
            assert ws.launches % ws.P == 0 and ws.pub_act_cnt == ws.P * (ws.launches // ws.P)
            clear_error_state(ws)
        else:
            res = run_launch(ws, rnd, launch_id, L, stack)
            assert set(res.values()) == {"done"}, (launch_id, res)


def test_the_timeout_hook_fails_every_block_then_the_next_launch_runs():
    """The workspace test hook (every reader expects a later epoch): no wait
    can complete, every block gives up after its bounded wait and leaves; with
    the error state cleared the next stack launch completes."""
    rnd = random.Random(7)
    ws = Ws(P=3)
    run_launch(ws, rnd, 0, 3, True)
    ws.hook = 1
    res = run_launch(ws, rnd, 1, 3, True, budget=200)
    assert set(res.values()) == {"failed"} and ws.status == 1
    clear_error_state(ws)
    res = run_launch(ws, rnd, 2, 4, True)
    assert set(res.values()) == {"done"}
    res = run_launch(ws, rnd, 3, 1, False)
    assert set(res.values()) == {"done"}


@pytest.mark.parametrize("mutate", ["same_epoch", "no_launch_tail"])
def test_the_model_catches_a_broken_protocol(mutate):
    """The check has teeth: with either planted mistake some interleaving of
    mixed launches accepts a word of another layer or launch."""
    caught = False
    for seed in range(40):
        rnd = random.Random(1000 + seed)
        ws = Ws(P=3)
        try:
            for launch_id in range(10):
                stack = rnd.random() < 0.7
                L = rnd.choice([2, 3]) if stack else 1
                res = run_launch(ws, rnd, launch_id, L, stack, budget=300, mutate=mutate)
                if set(res.values()) != {"done"}:
                    break  # a wait that never completes: the mistake shows as a hang instead
        except AssertionError:
            caught = True
            break
    assert caught
