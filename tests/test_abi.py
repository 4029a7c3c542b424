"""The C-ABI library builds, loads and exports every entry point that
include/rollout.h declares.  CPU only: no compute calls."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "rollout.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(rollout_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def libpath():
    from rl_experience_collection_gb300 import build
    return build.build()


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("rollout_create", "rollout_run", "rollout_destroy", "rollout_status", "rollout_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    for name in _declared():
        assert hasattr(lib, name), name
    from rl_experience_collection_gb300 import binding
    assert set(binding.EXPORTS) == set(_declared())


def _declared_ppo():
    src = open(os.path.join(ROOT, "include", "ppo.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ppo_[a-z_]+)\s*\(", src)))


def test_library_exports_every_ppo_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    names = _declared_ppo()
    assert "ppo_update" in names and "ppo_create" in names
    for name in names:
        assert hasattr(lib, name), name
    from rl_experience_collection_gb300 import binding
    assert set(binding.PPO_EXPORTS) == set(names)


def test_ppo_hparams_field_order_matches_header():
    from rl_experience_collection_gb300 import binding
    src = open(os.path.join(ROOT, "include", "ppo.h")).read()
    body = src[src.index("typedef struct {"):src.index("} ppo_hparams;")]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"\b([a-z_0-9]+)\s*(?=[,;])", body.replace("typedef struct {", "").replace("float", ""))
    assert fields == [f for f, _ in binding.PpoHparams._fields_]


def test_binding_struct_matches_header_field_order():
    from rl_experience_collection_gb300 import binding
    src = open(os.path.join(ROOT, "include", "rollout.h")).read()
    body = src[src.index("typedef struct {"):src.index("} rollout_dims;")]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = []
    for decl in body.split(";"):
        decl = decl.strip().replace("typedef struct {", "").strip()
        if not decl:
            continue
        typ, rest = decl.split(None, 1)
        for name in rest.split(","):
            fields.append(name.strip().split("[")[0])
    assert fields == [f for f, _ in binding.RolloutDims._fields_]


def test_last_error_callable_without_gpu(libpath):
    from rl_experience_collection_gb300 import binding
    binding.lib()
    assert isinstance(binding.last_error(), str)


def _declared_per():
    src = open(os.path.join(ROOT, "include", "per.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(per_[a-z_]+)\s*\(", src)))


def test_library_exports_every_replay_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    names = _declared_per()
    assert {"per_create", "per_insert", "per_sample", "per_update_priorities", "per_destroy"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name
    from rl_experience_collection_gb300 import binding
    assert set(binding.PER_EXPORTS) == set(names)


def _declared_dqn():
    src = open(os.path.join(ROOT, "include", "dqn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dqn_[a-z_]+)\s*\(", src)))


def test_library_exports_every_dqn_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    names = _declared_dqn()
    assert {"dqn_create", "dqn_run", "dqn_destroy", "dqn_weight_count"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name
    from rl_experience_collection_gb300 import binding
    assert set(binding.DQN_EXPORTS) == set(names)
    from rl_experience_collection_gb300 import workloads as wl
    assert binding.lib().dqn_weight_count() == 2 * wl.dqn_net_params() + wl.dqn_cur_params()
