"""Seeded synthetic input generators shared by the oracle, the tests and the bench."""
