"""CPU oracle for fused PPO experience collection -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference legs may import this package.
"""
