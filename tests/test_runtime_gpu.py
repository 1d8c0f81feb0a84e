"""GPU checks of the runtime around the kernels: the kernels loaded are the sm_103a build, and
host threads may call the library at the same time on one device."""
import threading

import pytest
import torch

from attention_backward_fabwd_gb300 import api, build, fabwd as F, inputs

import fabwd_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    F.lib()


def test_kernels_loaded_are_the_sm103a_build():
    torch.cuda.set_device(0)
    assert F.fabwd_kernel_binary_version() == 103


@pytest.mark.parametrize("d", [128, 192])
def test_two_host_threads_on_one_device(d):
    # Each thread drives its own problem on its own stream of device 0; the first launch of a
    # kernel sets its shared-memory limit for the device, and both threads may get there first.
    # (A fresh process would be needed to race the very first launch; this checks that
    # concurrent calls are correct and report no error.)
    W = inputs.WORKLOADS
    cases = [inputs.sized(W["causal_s8192_d192_dv128"] if d == 192 else W["gqa_causal_s4096_d128"], N1=4, N2=2,
                          S1=260 + 70 * i, S2=260 + 70 * i, dout_std=1.0, seed=50 + i) for i in range(2)]
    pbs = [inputs.make_problem(w) for w in cases]
    refs = [tl.full_reference(pb) for pb in pbs]
    results, errors = [None, None], []

    def work(i):
        try:
            torch.cuda.set_device(0)
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                dev = torch.device("cuda", 0)
                args = [t.to(dev) for t in (pbs[i].q, pbs[i].k, pbs[i].v, pbs[i].dout, refs[i].attn_out, refs[i].lse)]
                for _ in range(3):
                    out = api.flash_attn_grad(*args, mask_mode=1, check_status=True)
                st.synchronize()
                results[i] = [t.cpu() for t in out]
        except Exception as e:  # reported below, in the main thread
            errors.append(e)

    th = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join(timeout=300)
    assert not errors, errors
    for i in range(2):
        for name, got, want in zip(("dq", "dk", "dv"), results[i], (refs[i].dq, refs[i].dk, refs[i].dv)):
            tl.assert_close(f"thread {i} {name}", got, want)
